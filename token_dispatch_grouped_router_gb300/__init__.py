"""GB300-native single-GPU MoE expert layer: router top-k, device route map,
rowwise dispatch, unpadded grouped SwiGLU GEMM on tcgen05 tensor cores,
combine, and the backward of every step, behind the C-ABI library libmoe."""
