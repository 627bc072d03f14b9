// bfloat16 instantiations of the fused residual add + RMSNorm + quant kernels.
#include "rq_norm_quant_launch.cuh"

RQ_INSTANTIATE_NORM_QUANT(rq::BF16)
