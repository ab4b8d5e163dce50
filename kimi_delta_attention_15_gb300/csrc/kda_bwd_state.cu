// Backward, state-side products of each chunk: one CTA per (chunk, head), all
// chunks in parallel. From the checkpoints S0^T (forward) and dS_L^T (backward
// scan), stored key-major by the scans, and Ut, dUt, dO of the chunk, with tcgen05 tf32 MMAs (M = 128 over
// the key channel k):
//   dQbar = scale dO S0            [c][k]
//   dW    = -dUt S0                [c][k]
//   dKbar = Ut dS_L                [c][k]
//   dAqk  = scale dO Ut^T          [i][j], kept for j <= i
//   dgam  = sum_v dS_L[v,k] S0[v,k]  (adjoint of exp(G_L) through the decayed state,
//                                    before the factor exp(G_L))
// These are the reverse mode of Ut = U - W S0^T, O = scale[(Q^*Gamma) S0^T + Aqk Ut],
// S_L = S0 diag(exp(G_L)) + Ut^T (K^*e^{G_L-G}).
#include "kda_internal.cuh"
#include "umma.cuh"

namespace kda {

namespace {
struct BStateSmem {
    uint8_t S0T[kTileDD];    // S0^T   [128 k][128 v]
    uint8_t DST[kTileDD];    // dS_L^T [128 k][128 v]
    uint8_t STK[kTileDD];    // rows 0..63: dO [c][v]; rows 64..127: dUt [c][v]
    uint8_t UT[kTileCK];     // Ut [64 c][128 v]
    uint64_t bar, barC, barM;
    uint32_t tmem;
};
}  // namespace

size_t bwd_state_smem_bytes() { return sizeof(BStateSmem) + 1024; }

__global__ void __launch_bounds__(256, 1)
    kda_bwd_state_kernel(const uint16_t* __restrict__ dO, int H, float scale, uint8_t* __restrict__ ws, Layout lay) {
    extern __shared__ uint8_t smem_raw[];
    BStateSmem& s = *reinterpret_cast<BStateSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (read_status(ws) != 0) return;
    const int chunk = blockIdx.x, h = blockIdx.y;
    const ChunkInfo ci = reinterpret_cast<const ChunkInfo*>(ws + lay.chunks)[chunk];
    if (ci.L <= 0) return;
    const int tid = threadIdx.x, warp = tid >> 5;
    const size_t tile = (size_t)chunk * H + h;
    const uint8_t* gS0 = ws + lay.s0 + tile * kTileDD;
    const uint8_t* gDS = ws + lay.ds + tile * kTileDD;
    const uint8_t* gUt = ws + lay.ut + tile * kTileCK;
    const uint8_t* gdU = ws + lay.dut + tile * kTileCK;

    if (warp == 0) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&s.bar, 1); mbar_init(&s.barC, 1); mbar_init(&s.barM, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // Ut and dUt (fp32) are used split into tf32 high and low parts, in two
    // passes over the same buffers: pass 1 with the high parts, pass 2 adds
    // the products with the low parts (S0, dS_L and dO are exact in tf32).
    auto load_u = [&](uint32_t) {
        if (tid == 0) {
            mbar_arrive_expect_tx(&s.bar, (uint32_t)(2 * kTileCK));
            bulk_g2s(s.UT, gUt, (uint32_t)kTileCK, &s.bar);
            for (int p = 0; p < 4; ++p)
                bulk_g2s(s.STK + p * (D * 128) + 64 * 128, gdU + p * (C * 128), C * 128, &s.bar);
        }
    };
    // to high (lo = false) or low (lo = true) tf32 parts, in place
    auto split_u = [&](bool lo) {
        for (int i = tid; i < C * D; i += blockDim.x) {
            float* a = reinterpret_cast<float*>(s.UT) + i;
            const int r = i >> 7, c = i & 127;   // any bijection over the 64 x 128 elements
            float* b = reinterpret_cast<float*>(s.STK + panel_off(64 + r, c, D));
            const float x = *a, y = *b;
            *a = lo ? tf32_round(x - tf32_round(x)) : tf32_round(x);
            *b = lo ? tf32_round(y - tf32_round(y)) : tf32_round(y);
        }
    };
    load_u(0);
    // checkpoints S0^T and dS_L^T arrive in operand layout by bulk copy
    if (tid == 0) {
        mbar_arrive_expect_tx(&s.barC, (uint32_t)(2 * kTileDD));
        bulk_g2s(s.S0T, gS0, (uint32_t)kTileDD, &s.barC);
        bulk_g2s(s.DST, gDS, (uint32_t)kTileDD, &s.barC);
    }
    // dO rows 0..63 of the stack (bf16 values are exact in tf32; the scale is applied on readback)
    {
        const int v = tid & (D - 1), half = tid >> 7;
        uint16_t dov[C / 2];
#pragma unroll
        for (int i = 0; i < C / 2; ++i) {
            const int c = half * (C / 2) + i;
            dov[i] = c < ci.L ? dO[((size_t)(ci.t0 + c) * H + h) * D + v] : (uint16_t)0;
        }
#pragma unroll
        for (int i = 0; i < C / 2; ++i)
            *reinterpret_cast<float*>(s.STK + panel_off(half * (C / 2) + i, v, D)) = bf2f(dov[i]);
    }
    const uint32_t tm = s.tmem;
    bool ok = mbar_wait(&s.bar, 0) && mbar_wait(&s.barC, 0);
    ok = __syncthreads_and(ok);
    if (ok) split_u(false);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t aS = smem_u32(s.S0T), aD = smem_u32(s.DST), aK = smem_u32(s.STK), bU = smem_u32(s.UT);
    const uint32_t id128 = idesc_tf32(128, 128, 0, 0), id64 = idesc_tf32(128, 64, 0, 0);
    if (tid == 0 && ok) {
        // [dQbar / scale | dUt S0]^T = S0^T [dO ; dUt]^T  -> cols 0..127
        for (int ks = 0; ks < D / 8; ++ks)
            umma_tf32(tm + 0, desc_kmajor(aS, D, ks), desc_kmajor(aK, D, ks), id128, ks > 0);
        // dKbar^T = dS_L^T Ut^T                            -> cols 128..191
        for (int ks = 0; ks < D / 8; ++ks)
            umma_tf32(tm + 128, desc_kmajor(aD, D, ks), desc_kmajor(bU, C, ks), id64, ks > 0);
        // dS_L^T S0 (diagonal used)                         -> cols 256..383
        for (int ks = 0; ks < D / 8; ++ks)
            umma_tf32(tm + 256, desc_kmajor(aD, D, ks), desc_kmajor(aS, D, ks), id128, ks > 0);
        // [dO ; dUt] Ut^T (rows 0..63 used, x scale)      -> cols 384..447
        for (int ks = 0; ks < D / 8; ++ks)
            umma_tf32(tm + 384, desc_kmajor(aK, D, ks), desc_kmajor(bU, C, ks), id64, ks > 0);
        umma_commit(&s.barM);
    }
    ok = (ok && mbar_wait(&s.barM, 0));
    ok = __syncthreads_and(ok);
    // pass 2: the low parts of Ut and dUt
    if (ok) {
        tc_fence_after();
        load_u(1);
        ok = mbar_wait(&s.bar, 1);
        ok = __syncthreads_and(ok);
    }
    if (ok) split_u(true);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && ok) {
        // (dUt_lo S0)^T                                     -> cols 64..127
        for (int ks = 0; ks < D / 8; ++ks)
            umma_tf32(tm + 64, desc_kmajor(aS, D, ks), desc_kmajor(aK, D, ks, 64), id64, 1);
        for (int ks = 0; ks < D / 8; ++ks)
            umma_tf32(tm + 128, desc_kmajor(aD, D, ks), desc_kmajor(bU, C, ks), id64, 1);
        for (int ks = 0; ks < D / 8; ++ks)
            umma_tf32(tm + 384, desc_kmajor(aK, D, ks), desc_kmajor(bU, C, ks), id64, 1);
        umma_commit(&s.barM);
    }
    ok = (ok && mbar_wait(&s.barM, 1));
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (ok) {
        // warp w reads TMEM lanes 32 (w % 4) .. +31; warps w and w + 4 split the columns
        const int kq = (warp & 3) * 32 + (tid & 31);   // lane = key channel k (or row i for dAqk)
        const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
        const int c0 = (warp >> 2) * 32;
        uint8_t* bg = ws + lay.bg + tile * BgOff::BYTES;
        float* gdQ = reinterpret_cast<float*>(bg + BgOff::DQB);
        float* gdW = reinterpret_cast<float*>(bg + BgOff::DW);
        float* gdK = reinterpret_cast<float*>(bg + BgOff::DKB);
        float* gdA = reinterpret_cast<float*>(bg + BgOff::DAQK);
        float* gdG = reinterpret_cast<float*>(bg + BgOff::DGAM);
        {
            float r[32];
            tmem_ld32(tm + lb + c0, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) gdQ[(c0 + j) * D + kq] = scale * r[j];
            tmem_ld32(tm + lb + 64 + c0, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) gdW[(c0 + j) * D + kq] = -r[j];
            tmem_ld32(tm + lb + 128 + c0, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) gdK[(c0 + j) * D + kq] = r[j];
        }
        if (warp < 4) {
            float r[32];
            tmem_ld32(tm + lb + 256 + warp * 32, r);
            float dg = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) dg = (j == (tid & 31)) ? r[j] : dg;
            gdG[kq] = dg;
        }
        if ((warp & 3) < 2) {
            const int i = kq;
            float r[32];
            tmem_ld32(tm + lb + 384 + c0, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) gdA[i * C + c0 + j] = (c0 + j <= i) ? scale * r[j] : 0.0f;
        }
    } else {
        raise_status(ws, KDA_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace kda
