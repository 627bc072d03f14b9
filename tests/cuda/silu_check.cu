// silu_check.cu -- checks of the library's SiLU gate (rq::silu_fast,
// rq::silu_near_tie, rq::silu_gate8), built and run by tests/test_gpu_gated.py.
//
//  1. Over every finite fp32 z >= -87 (the inputs the fast path serves): the
//     largest distance, counted in fp32 bit patterns (ulps), between
//     silu_fast(z) and z / (1 + e^-z) evaluated in double precision and
//     rounded once to fp32.  rq::kSiluUlps, the window of the near-tie test,
//     must bound it.
//  2. For bf16 and fp16, the gate dt(silu(z)) that silu_gate8 gives for every
//     one of the 65,536 bit patterns z, and the gates that the gated kernels
//     take from their shared-memory tables (gate8_bf16, gate8_fp16), written
//     to the file named by argv[1] (65,536 bf16 gates, 65,536 fp16 gates,
//     65,536 bf16 table gates, 65,536 fp16 table gates) for the test to
//     compare with the oracle's, and how many of the patterns with |z| <= 8
//     took the exact path.
#include <cstdio>

#include "rq_device.cuh"

__device__ unsigned int g_max_bits;
__device__ unsigned int g_slow[2];

__device__ float ref_silu(float z)
{
    const double d = (double)z;
    return (float)(d / (1.0 + exp(-d)));
}

// fp32 bit pattern as a signed position on the number line (+0 and -0 both 0)
__device__ long long ordinal(float v)
{
    const unsigned b = __float_as_uint(v);
    const long long m = b & 0x7FFFFFFFu;
    return (b >> 31) ? -m : m;
}

__global__ void check_fast()
{
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < (1ull << 32);
         i += (unsigned long long)gridDim.x * blockDim.x) {
        const float z = __uint_as_float((unsigned)i);
        if (!isfinite(z) || z < -87.0f) continue;
        const long long d = ordinal(rq::silu_fast(z)) - ordinal(ref_silu(z));
        const unsigned long long a = d < 0 ? -d : d;
        if (a) atomicMax(&g_max_bits, a > 0xFFFFFFFFull ? 0xFFFFFFFFu : (unsigned)a);
    }
}

// thread i: the 8 patterns 8i .. 8i + 7 of one dtype
template <typename DT>
__global__ void gates(unsigned short *out, int which)
{
    const unsigned i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 65536u / 8) return;
    uint4 zv;
    const unsigned b = 8 * i;
    zv.x = b | ((b + 1) << 16);
    zv.y = (b + 2) | ((b + 3) << 16);
    zv.z = (b + 4) | ((b + 5) << 16);
    zv.w = (b + 6) | ((b + 7) << 16);
    const uint4 g = rq::silu_gate8<DT>(zv);
    const unsigned w[4] = {g.x, g.y, g.z, g.w};
    float z[8];
    rq::unpack8<DT>(zv, z);
    for (int e = 0; e < 8; ++e) {
        out[b + e] = (unsigned short)(w[e / 2] >> (16 * (e & 1)));
        if (fabsf(z[e]) <= 8.0f && rq::silu_near_tie<DT>(rq::silu_fast(z[e]), z[e]))
            atomicAdd(&g_slow[which], 1u);
    }
}

// the gated kernel's bf16 path: table built in shared memory, then lookups
// (thread i: the 8 patterns 8i .. 8i + 7)
__global__ void table_gates(unsigned short *out)
{
    __shared__ __align__(16) uint16_t tab[2 * rq::kGateHalf];
    rq::gate_table_fill(tab);
    __syncthreads();
    const unsigned i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 65536u / 8) return;
    const unsigned b = 8 * i;
    const uint4 zv = make_uint4(b | ((b + 1) << 16), (b + 2) | ((b + 3) << 16),
                                (b + 4) | ((b + 5) << 16), (b + 6) | ((b + 7) << 16));
    const uint4 g = rq::gate8_bf16(zv, tab);
    const unsigned w[4] = {g.x, g.y, g.z, g.w};
    for (int e = 0; e < 8; ++e) out[b + e] = (unsigned short)(w[e / 2] >> (16 * (e & 1)));
}

// the same for fp16: its table in dynamic shared memory
__global__ void table_gates_fp16(unsigned short *out)
{
    extern __shared__ __align__(16) uint16_t tab16[];
    rq::gate_table_fill_fp16(tab16);
    __syncthreads();
    const unsigned i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= 65536u / 8) return;
    const unsigned b = 8 * i;
    const uint4 zv = make_uint4(b | ((b + 1) << 16), (b + 2) | ((b + 3) << 16),
                                (b + 4) | ((b + 5) << 16), (b + 6) | ((b + 7) << 16));
    const uint4 g = rq::gate8_fp16(zv, tab16);
    const unsigned w[4] = {g.x, g.y, g.z, g.w};
    for (int e = 0; e < 8; ++e) out[b + e] = (unsigned short)(w[e / 2] >> (16 * (e & 1)));
}

int main(int argc, char **argv)
{
    if (argc < 2) {
        std::printf("usage: silu_check <gates output file>\n");
        return 2;
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    unsigned short *d_out = nullptr;
    const int tab16_bytes = 2 * rq::kGateHalfF16 * 2;
    if (cudaFuncSetAttribute(table_gates_fp16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tab16_bytes) != cudaSuccess ||
        cudaMalloc(&d_out, 4 * 65536 * sizeof(unsigned short)) != cudaSuccess) {
        std::printf("error: cudaMalloc\n");
        return 2;
    }
    check_fast<<<sms * 8, 256>>>();
    gates<rq::BF16><<<32, 256>>>(d_out, 0);
    gates<rq::FP16><<<32, 256>>>(d_out + 65536, 1);
    table_gates<<<32, 256>>>(d_out + 2 * 65536);
    table_gates_fp16<<<32, 256, tab16_bytes>>>(d_out + 3 * 65536);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        std::printf("error %s\n", cudaGetErrorString(e));
        return 2;
    }
    static unsigned short h[4 * 65536];
    unsigned int mx = 0, slow[2] = {0, 0};
    cudaMemcpy(h, d_out, sizeof(h), cudaMemcpyDeviceToHost);
    cudaMemcpyFromSymbol(&mx, g_max_bits, sizeof(mx));
    cudaMemcpyFromSymbol(slow, g_slow, sizeof(slow));
    cudaFree(d_out);
    FILE *f = std::fopen(argv[1], "wb");
    if (!f || std::fwrite(h, sizeof(h), 1, f) != 1) {
        std::printf("error: cannot write %s\n", argv[1]);
        return 2;
    }
    std::fclose(f);
    std::printf("silu max_bits %u window %d slow_bf16 %u slow_fp16 %u\n", mx, rq::kSiluUlps, slow[0],
                slow[1]);
    return 0;
}
