"""GB300-native split-K W4A16-g128 projection matmul.

The product is the C-ABI library libqmm.so (include/qmm.h), built in-tree by
``split_w4a16_quantized_gb300.build``; ``split_w4a16_quantized_gb300.qmm`` is
its Python binding and ``split_w4a16_quantized_gb300.inputs`` the seeded
synthetic workload generator.
"""
