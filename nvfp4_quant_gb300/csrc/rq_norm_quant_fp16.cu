// float16 instantiations of the fused residual add + RMSNorm + quant kernels.
#include "rq_norm_quant_launch.cuh"

#ifdef RQ_MODE
RQ_INSTANTIATE_MODE(rq::FP16, RQ_MODE)
#else
RQ_INSTANTIATE_NORM_QUANT(rq::FP16)
#endif
