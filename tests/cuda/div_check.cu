// div_check.cu -- compares the library's shared-divisor division (rq::div_by,
// Markstein's correction step) with CUDA's correctly rounded __fdiv_rn over
// every finite fp32 dividend, for each divisor given on the command line.
// Prints, per divisor: the fp32 quotients that differ where the reference
// quotient has magnitude in [2^-40, 2^20), the E4M3 codes (satfinite)
// that differ anywhere, NaN and infinite dividends included, and, for the
// packed two-wide magnitude version the Q/K kernel uses (rq::div_mag_by2 on
// the pair (a, -a), with the sign of a put back on the E4M3 code byte), the
// non-NaN dividends whose magnitudes are not bit for bit |div_by(a)| or whose
// codes are not the scalar version's.  Built and run by tests/test_gpu_division.py.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "rq_device.cuh"

__device__ unsigned long long g_quot_diff, g_code_diff, g_pack_diff;
__device__ unsigned int g_first_bad;

__global__ void check(float b)
{
    const rq::Divisor d(b);
    const unsigned long long n = 1ull << 32;
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n;
         i += (unsigned long long)gridDim.x * blockDim.x) {
        const unsigned int bits = (unsigned int)i;
        const float a = __uint_as_float(bits);
        const float ref = __fdiv_rn(a, b);
        const float got = d.fast ? rq::div_by<true>(a, d) : rq::div_by<false>(a, d);
        const float m = fabsf(ref);
        if (m >= 0x1p-40f && m < 0x1p20f && __float_as_uint(ref) != __float_as_uint(got)) {
            if (atomicAdd(&g_quot_diff, 1ull) == 0) g_first_bad = bits;
        }
        if ((rq::e4m3x2(ref, 0.0f) & 0xFF) != (rq::e4m3x2(got, 0.0f) & 0xFF))
            atomicAdd(&g_code_diff, 1ull);
        const float na = __uint_as_float(bits ^ 0x80000000u);
        const float2 g2 = d.fast ? rq::div_mag_by2<true>(make_float2(a, na), d)
                                 : rq::div_mag_by2<false>(make_float2(a, na), d);
        if (!isnan(a)) {
            const unsigned int mag = __float_as_uint(got) & 0x7FFFFFFFu;
            const unsigned int code = (rq::e4m3x2(g2.x, 0.0f) & 0xFFu) | ((bits >> 24) & 0x80u);
            if (__float_as_uint(g2.x) != mag || __float_as_uint(g2.y) != mag ||
                code != (rq::e4m3x2(got, 0.0f) & 0xFFu))
                atomicAdd(&g_pack_diff, 1ull);
        }
    }
}

int main(int argc, char **argv)
{
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    for (int k = 1; k < argc; ++k) {
        const float b = strtof(argv[k], nullptr);
        unsigned long long zero = 0;
        unsigned int z = 0;
        cudaMemcpyToSymbol(g_quot_diff, &zero, sizeof(zero));
        cudaMemcpyToSymbol(g_code_diff, &zero, sizeof(zero));
        cudaMemcpyToSymbol(g_pack_diff, &zero, sizeof(zero));
        cudaMemcpyToSymbol(g_first_bad, &z, sizeof(z));
        check<<<sms * 8, 256>>>(b);
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            std::printf("error %s\n", cudaGetErrorString(e));
            return 2;
        }
        unsigned long long qd = 0, cd = 0, pd = 0;
        unsigned int first = 0;
        cudaMemcpyFromSymbol(&qd, g_quot_diff, sizeof(qd));
        cudaMemcpyFromSymbol(&cd, g_code_diff, sizeof(cd));
        cudaMemcpyFromSymbol(&pd, g_pack_diff, sizeof(pd));
        cudaMemcpyFromSymbol(&first, g_first_bad, sizeof(first));
        std::printf("divisor %.9g quotient_diffs %llu code_diffs %llu first 0x%08x packed_diffs %llu\n", b, qd,
                    cd, first, pd);
    }
    return 0;
}
