// Diagnostic kernel for the tcgen05 building blocks: one CTA computes
// D[128 x N] = A[128 x Kd] * B[N x Kd]^T with kind::tf32 operands laid out in
// shared memory K-major or MN-major, then reads D back from TMEM, writes it
// back scaled through tcgen05.st and reads it again. It checks the operand
// descriptors and the TMEM data path used by the KDA kernels.
#include "umma.cuh"
#include "kda_internal.cuh"

namespace kda {

__global__ void __launch_bounds__(128, 1)
    umma_selftest_kernel(int a_mn, int b_mn, int N, int Kd, const float* __restrict__ A,
                         const float* __restrict__ B, float* __restrict__ D) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;                       // 128 * Kd floats
    uint8_t* sB = smem + 128 * Kd * 4;        // N * Kd floats
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int idx = tid; idx < 128 * Kd; idx += blockDim.x) {
        const int m = idx / Kd, k = idx % Kd;
        const float x = tf32_round(A[idx]);
        const uint32_t off = a_mn ? panel_off(k, m, Kd) : panel_off(m, k, 128);
        *reinterpret_cast<float*>(sA + off) = x;
    }
    for (int idx = tid; idx < N * Kd; idx += blockDim.x) {
        const int n = idx / Kd, k = idx % Kd;
        const float x = tf32_round(B[idx]);
        const uint32_t off = b_mn ? panel_off(k, n, Kd) : panel_off(n, k, N);
        *reinterpret_cast<float*>(sB + off) = x;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_base;
    if (tid == 0) {
        const uint32_t idesc = idesc_tf32(128, N, a_mn, b_mn);
        const uint32_t aa = smem_u32(sA), ba = smem_u32(sB);
        for (int s = 0; s < Kd / 8; ++s) {
            const uint64_t ad = a_mn ? desc_mnmajor(aa, Kd, s) : desc_kmajor(aa, 128, s);
            const uint64_t bd = b_mn ? desc_mnmajor(ba, Kd, s) : desc_kmajor(ba, N, s);
            umma_tf32(tm, ad, bd, idesc, s > 0 ? 1u : 0u);
        }
        umma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0);
    tc_fence_after();
    const int row = warp * 32 + lane;
    for (int c0 = 0; c0 < N; c0 += 32) {
        float v[32];
        tmem_ld32(tmem_addr(tm, warp * 32, c0), v);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            D[row * N + c0 + j] = ok ? v[j] : __int_as_float(0x7fc00000);
            v[j] = 2.0f * v[j] + (float)row;
        }
        tmem_st32(tmem_addr(tm, warp * 32, c0), v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    for (int c0 = 0; c0 < N; c0 += 32) {
        float v[32];
        tmem_ld32(tmem_addr(tm, warp * 32, c0), v);
#pragma unroll
        for (int j = 0; j < 32; ++j) D[128 * N + row * N + c0 + j] = v[j];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// Waits on an mbarrier that nothing will ever complete, with a limit of
// limit_ns, then reports KDA_ERR_TIMEOUT in the status word at `status_word`
// the same way the KDA kernels do. Exercises the timeout path without hanging.
__global__ void wait_timeout_kernel(uint64_t limit_ns, uint8_t* status_word) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    bool ok = mbar_wait(&bar, 0, limit_ns);   // nobody arrives
    ok = __syncthreads_and(ok);
    if (!ok && threadIdx.x == 0) raise_status(status_word, KDA_ERR_TIMEOUT);
}

// Both tf32 roundings of each input: the library's (tf32_round, integer operations)
// and the hardware conversion cvt.rna.tf32.f32 it stands in for.
__global__ void tf32_round_kernel(const float* __restrict__ in, float* __restrict__ out,
                                  float* __restrict__ ref, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float x = in[i];
        uint32_t r;
        asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
        out[i] = tf32_round(x);
        ref[i] = __uint_as_float(r);
    }
}

}  // namespace kda

extern "C" int kda_diag_tf32_round(const float* in, float* out, float* ref, long long n, void* stream) {
    if (n < 0) return KDA_ERR_SHAPE;
    if (n == 0) return KDA_OK;
    if (!in || !out || !ref) return KDA_ERR_NULL;
    const long long blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    kda::tf32_round_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(in, out, ref, (int64_t)n);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" int kda_diag_wait_timeout(unsigned long long limit_ns, void* workspace, void* stream) {
    if (!workspace) return KDA_ERR_NULL;
    if (limit_ns == 0 || limit_ns > 1000000000ull) return KDA_ERR_UNSUPPORTED;
    kda::wait_timeout_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(limit_ns, static_cast<uint8_t*>(workspace));
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" int kda_diag_umma_selftest(int a_mn, int b_mn, int N, int Kd, const float* A, const float* B,
                                      float* D, void* stream) {
    if (N < 16 || N > 256 || (N % 16) || Kd < 8 || Kd > 128 || (Kd % 32)) return KDA_ERR_SHAPE;
    if (a_mn || b_mn) return KDA_ERR_UNSUPPORTED;   // kind::tf32 takes K-major operands only
    if (!A || !B || !D) return KDA_ERR_NULL;
    const size_t smem = (size_t)(128 + N) * Kd * 4 + 1024;
    cudaError_t e = cudaFuncSetAttribute(kda::umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    kda::umma_selftest_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(a_mn, b_mn, N, Kd, A, B, D);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
