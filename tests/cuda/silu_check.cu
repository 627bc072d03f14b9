// silu_check.cu -- error of the library's fp32 SiLU (rq::silu_f32) against
// the correctly rounded fp32 value of z / (1 + e^-z), taken from a double
// precision evaluation, over every finite fp32 input z.  Prints the largest
// error in fp32 ulps (of the reference) over normal results and the number
// of those more than 1, 2 and 4 ulps off; for bf16 and fp16, how many of the
// 65,536 dtype values of z give a different dtype-rounded SiLU; and the
// largest error, in units of the smallest subnormal, over subnormal results.  Built and run by
// tests/test_gpu_gated.py.
#include <cstdio>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "rq_device.cuh"

__device__ unsigned long long g_over[3];
__device__ unsigned int g_max_ulp, g_max_ulp_sub;
__device__ unsigned int g_dt_diff[2];

__device__ float ref_silu(float z)
{
    const double d = (double)z;
    return (float)(d / (1.0 + exp(-d)));
}

__device__ float ulp_of(float v)
{
    const float a = fabsf(v);
    if (a < 0x1p-126f) return 0x1p-149f;
    return __int_as_float(__float_as_int(a) & 0x7F800000) * 0x1p-23f;
}

__global__ void check_all()
{
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < (1ull << 32);
         i += (unsigned long long)gridDim.x * blockDim.x) {
        const float z = __uint_as_float((unsigned)i);
        if (!isfinite(z)) continue;
        const float ref = ref_silu(z), got = rq::silu_f32(z);
        if (__float_as_uint(ref) == __float_as_uint(got)) continue;
        const float err = fabsf(got - ref) / ulp_of(ref);
        const unsigned e = err > 1e9f ? 1000000000u : (unsigned)ceilf(err);
        if (fabsf(ref) < 0x1p-126f) {  // subnormal results: counted apart
            atomicMax(&g_max_ulp_sub, e);
            continue;
        }
        atomicMax(&g_max_ulp, e);
        if (err > 1.0f) atomicAdd(&g_over[0], 1ull);
        if (err > 2.0f) atomicAdd(&g_over[1], 1ull);
        if (err > 4.0f) atomicAdd(&g_over[2], 1ull);
    }
}

__global__ void check_dtypes()
{
    const unsigned b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= 65536u) return;
    const unsigned short u = (unsigned short)b;
    const float zb = __bfloat162float(__ushort_as_bfloat16(u));
    if (isfinite(zb) &&
        __bfloat16_as_ushort(__float2bfloat16_rn(ref_silu(zb))) !=
            __bfloat16_as_ushort(__float2bfloat16_rn(rq::silu_f32(zb))))
        atomicAdd(&g_dt_diff[0], 1u);
    const float zh = __half2float(__ushort_as_half(u));
    if (isfinite(zh) &&
        __half_as_ushort(__float2half_rn(ref_silu(zh))) != __half_as_ushort(__float2half_rn(rq::silu_f32(zh))))
        atomicAdd(&g_dt_diff[1], 1u);
}

int main()
{
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    check_all<<<sms * 8, 256>>>();
    check_dtypes<<<256, 256>>>();
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        std::printf("error %s\n", cudaGetErrorString(e));
        return 2;
    }
    unsigned long long over[3];
    unsigned int mx, mxs, dd[2];
    cudaMemcpyFromSymbol(over, g_over, sizeof(over));
    cudaMemcpyFromSymbol(&mx, g_max_ulp, sizeof(mx));
    cudaMemcpyFromSymbol(&mxs, g_max_ulp_sub, sizeof(mxs));
    cudaMemcpyFromSymbol(dd, g_dt_diff, sizeof(dd));
    std::printf("silu max_ulp %u over1 %llu over2 %llu over4 %llu bf16_diff %u fp16_diff %u subnormal_max_ulp %u\n",
                mx, over[0], over[1], over[2], dd[0], dd[1], mxs);
    return 0;
}
