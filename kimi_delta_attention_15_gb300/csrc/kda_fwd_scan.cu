// Forward state scan: one CTA per (sequence, head), chunks in order. The fp32
// state S (V x K = 128 x 128, value-first) lives in tensor memory (lane v =
// value row, column k = key channel). Per chunk, with the intra-chunk images
// W, Q^*Gamma, (K^*e^{G_L-G})^T, Aqk, U, exp(G_L):
//   Ut^T = U^T - S0 W^T                  (tcgen05, M=128 N=64 K=128)
//   O^T  = S0 (Q^*Gamma)^T + Ut^T Aqk^T  (tcgen05)
//   S_L  = S0 diag(exp(G_L)) + Ut^T (K^*e^{G_L-G})
//   o    = scale * O
// (chunk form of S_t = S_{t-1} diag(e^{g_t}) (I - b k^ k^T) + b v k^T,
//  o_t = scale S_t q^_t; flashinfer "kda_backward" contract). S0 of every
// chunk, rounded to tf32 as the MMAs use it, is checkpointed to the
// workspace for the backward as S0^T (key-major panels, the operand layout the
// backward's state products use), together with Ut (fp32).
// The MMAs with S0 read it from a tf32 copy in tensor memory (A operand in
// TMEM), which leaves shared memory for two W, Q^*Gamma buffers: those operands
// are requested two chunks ahead. Products that share their A operand run as
// one wide MMA over stacked B operands (panels interleaved in shared memory):
//   [Ut^T | O^T]   = S0 [W ; Q^*Gamma]^T                 (N = 128)
//   [O^T | S_L]   += Ut^T [Aqk ; (K^*e^{G_L-G})^T]^T     (N = 192)
// so TMEM holds Ut^T (columns 0..63), O^T (64..127), S (128..255), tf32 S0 (256..383).
#include "kda_internal.cuh"
#include "umma.cuh"

namespace kda {

namespace {
struct ScanSmem {
    // operand tiles, 1024-byte aligned (panels)
    // [W ; QB] as one 128-row operand: panel p = W rows (8 KB) then QB rows (8 KB); by chunk parity
    uint8_t WQ[2][2 * kTileCK];
    // [Aqk ; KBT] as one 192-row operand: panel p = Aqk rows (8 KB) then KBT rows (16 KB)
    uint8_t AK[kTileCK + kTileCC];
    uint8_t UT[kTileCK];       // [128 v][64 c]; between the state update and the next
                               // chunk's Ut also the bf16 output rows [64 i][128 v]
    float gam[D];
    uint64_t barA[2], barB, barM1, barM2;
    uint32_t tmem;
};
}  // namespace

size_t fwd_scan_smem_bytes() { return sizeof(ScanSmem) + 1024; }

__global__ void __launch_bounds__(256, 1)
    kda_fwd_scan_kernel(const float* __restrict__ h0, uint16_t* __restrict__ o, float* __restrict__ hT, int H,
                        float scale, uint8_t* __restrict__ ws, Layout lay) {
    extern __shared__ uint8_t smem_raw[];
    ScanSmem& s = *reinterpret_cast<ScanSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (read_status(ws) != 0) return;
    const int h = blockIdx.x;
    const int n = reinterpret_cast<const int*>(ws + lay.seq_order)[blockIdx.y];
    const int cf = reinterpret_cast<const int*>(ws + lay.seq_first)[n];
    const int cl = reinterpret_cast<const int*>(ws + lay.seq_first)[n + 1];
    const ChunkInfo* chunks = reinterpret_cast<const ChunkInfo*>(ws + lay.chunks);
    const int tid = threadIdx.x, warp = tid >> 5;
    // threads v and v + 128 own state row v (TMEM lane v) and split its columns
    const int v = tid & (D - 1), half = tid >> 7;
    const size_t sidx = ((size_t)n * H + h) * D * D;

    if (warp == 0) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&s.barA[0], 1); mbar_init(&s.barA[1], 1); mbar_init(&s.barB, 1); mbar_init(&s.barM1, 1); mbar_init(&s.barM2, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s.tmem;
    const uint32_t tUT = tm, tOT = tm + 64, tS = tm + 128, tS0 = tm + 256;   // tS0: tf32 copy of S0
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    // initial state into TMEM
    for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
        float r[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {   // a row per lane: 16-byte loads
            const float4 x = h0 ? *reinterpret_cast<const float4*>(h0 + sidx + (size_t)v * D + c0 + j)
                                : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            r[j] = x.x; r[j + 1] = x.y; r[j + 2] = x.z; r[j + 3] = x.w;
        }
        tmem_st32(tS + lane_base + c0, r);
    }

    // W, QB of chunk cf + i go to buffer i & 1 and complete phase (i >> 1) of barA[i & 1]
    auto issue_A = [&](int chunk) {
        const int b = (chunk - cf) & 1;
        const uint8_t* img = ws + lay.img + ((size_t)chunk * H + h) * ImgOff::BYTES;
        mbar_arrive_expect_tx(&s.barA[b], (uint32_t)(2 * kTileCK));
        for (int p = 0; p < 4; ++p) {
            bulk_g2s(s.WQ[b] + p * 2 * C * 128, img + ImgOff::W + p * C * 128, C * 128, &s.barA[b]);
            bulk_g2s(s.WQ[b] + p * 2 * C * 128 + C * 128, img + ImgOff::QB + p * C * 128, C * 128, &s.barA[b]);
        }
    };
    auto issue_B = [&](int chunk) {
        const uint8_t* img = ws + lay.img + ((size_t)chunk * H + h) * ImgOff::BYTES;
        mbar_arrive_expect_tx(&s.barB, (uint32_t)(kTileCK + kTileCC));
        for (int p = 0; p < 2; ++p) {
            bulk_g2s(s.AK + p * (C + D) * 128, img + ImgOff::AQK + p * C * 128, C * 128, &s.barB);
            bulk_g2s(s.AK + p * (C + D) * 128 + C * 128, img + ImgOff::KBT + p * D * 128, D * 128, &s.barB);
        }
    };
    int a_issued = 0, b_issued = 0, a_done = 0, b_done = 0;   // bulk groups (thread 0), in chunk order
    if (tid == 0 && cf < cl) {
        issue_A(cf);
        issue_B(cf);
        a_issued = b_issued = 1;
        if (cf + 1 < cl) { issue_A(cf + 1); a_issued = 2; }
    }

    bool ok = true;
    const uint32_t idN128 = idesc_tf32(128, 128, 0, 0);
    const uint32_t idN192 = idesc_tf32(128, 192, 0, 0);
    // per-chunk scalars are fetched one chunk ahead
    ChunkInfo ci_next = cf < cl ? chunks[cf] : ChunkInfo{0, 0, 0, 0};
    float gam_next = cf < cl ? reinterpret_cast<const float*>(ws + lay.img + ((size_t)cf * H + h) * ImgOff::BYTES +
                                                              ImgOff::GAML)[v]
                             : 0.0f;
    // output rows staged in s.UT wait for the next loop-top barrier, then go out as one
    // bulk store per token row (threads 128..191, row tid - 128)
    uint16_t* const ost = reinterpret_cast<uint16_t*>(s.UT);
    const bool o_thread = tid >= 128 && tid < 128 + C;
    int o_t0 = 0, o_L = 0;
    auto store_o_rows = [&]() {
        if (o_thread && tid - 128 < o_L) {
            bulk_s2g(o + ((size_t)(o_t0 + tid - 128) * H + h) * D, ost + (tid - 128) * D, (uint32_t)(2 * D));
            bulk_commit();
        }
        o_L = 0;
    };
    for (int chunk = cf; chunk < cl && ok; ++chunk) {
        const uint32_t par = (uint32_t)((chunk - cf) & 1);
        const ChunkInfo ci = ci_next;
        const size_t tile = (size_t)chunk * H + h;
        const uint8_t* img = ws + lay.img + tile * ImgOff::BYTES;
        const float* gU = reinterpret_cast<const float*>(img + ImgOff::U);
        if (half == 0) s.gam[v] = gam_next;
        if (chunk + 1 < cl) {
            ci_next = chunks[chunk + 1];
            gam_next = reinterpret_cast<const float*>(img + (size_t)H * ImgOff::BYTES + ImgOff::GAML)[v];  // chunk + 1
        }
        __syncthreads();
        store_o_rows();

        // S0: TMEM -> registers -> tf32 copy in TMEM (the MMA operand), and its transpose
        // S0^T [k][v] to the workspace checkpoint; decayed state back to TMEM
        // (both 32-column halves in flight at once: one wait for the loads, one for the stores)
        uint8_t* gS0T = ws + lay.s0 + tile * kTileDD;
        {
            const int cb = 64 * half;
            uint32_t r0[32], r1[32], q0[32], q1[32];
            tmem_ld32_issue(tS + lane_base + cb, r0);
            tmem_ld32_issue(tS + lane_base + cb + 32, r1);
            tmem_wait_ld(r0);
            tmem_after_wait(r1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                q0[j] = tf32_round_bits(__uint_as_float(r0[j]));
                q1[j] = tf32_round_bits(__uint_as_float(r1[j]));
            }
            tmem_st32_issue(tS0 + lane_base + cb, q0);
            tmem_st32_issue(tS0 + lane_base + cb + 32, q1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                *reinterpret_cast<uint32_t*>(gS0T + panel_off(cb + j, v, D)) = q0[j];
                *reinterpret_cast<uint32_t*>(gS0T + panel_off(cb + 32 + j, v, D)) = q1[j];
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                r0[j] = __float_as_uint(__uint_as_float(r0[j]) * s.gam[cb + j]);
                r1[j] = __float_as_uint(__uint_as_float(r1[j]) * s.gam[cb + 32 + j]);
            }
            tmem_st32_issue(tS + lane_base + cb, r0);
            tmem_st32_issue(tS + lane_base + cb + 32, r1);
            tmem_wait_st(q0);
            tmem_after_wait(q1);
            tmem_after_wait(r0);
            tmem_after_wait(r1);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        const int ab = (chunk - cf) & 1;
        if (tid == 0) {
            if (!mbar_wait(&s.barA[ab], (uint32_t)(((chunk - cf) >> 1) & 1))) ok = false;
            else ++a_done;
            if (ok) {
                const uint32_t bwq = smem_u32(s.WQ[ab]);
                for (int ks = 0; ks < D / 8; ++ks)
                    umma_tf32_ta(tUT, tS0 + 8 * ks, desc_kmajor(bwq, 2 * C, ks), idN128, ks > 0);
                umma_commit(&s.barM1);
            }
        }
        // U column v of this chunk
        float u[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) u[c] = gU[(32 * half + c) * D + v];
        ok = mbar_wait(&s.barM1, par) && ok;
        if (o_thread) bulk_wait_read_all();   // s.UT is rewritten below
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0 && chunk + 2 < cl) { issue_A(chunk + 2); ++a_issued; }   // into this chunk's buffer

        // Ut^T = U^T - S0 W^T  -> tf32 operand [v][c]; Ut (fp32) -> workspace [c][v] panels
        uint8_t* gUt = ws + lay.ut + tile * kTileCK;
        {
            const int c0 = 32 * half;
            float r[32];
            tmem_ld32(tUT + lane_base + c0, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = u[j] - r[j];
#pragma unroll
            for (int j = 0; j < 32; ++j) *reinterpret_cast<float*>(gUt + panel_off(c0 + j, v, C)) = r[j];
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(s.UT + panel_off(v, c0 + j, D)) =
                    make_float4(tf32_round(r[j]), tf32_round(r[j + 1]), tf32_round(r[j + 2]), tf32_round(r[j + 3]));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            if (!mbar_wait(&s.barB, par)) ok = false;
            else ++b_done;
            if (ok) {
                const uint32_t a = smem_u32(s.UT), bak = smem_u32(s.AK);
                for (int ks = 0; ks < C / 8; ++ks)
                    umma_tf32(tOT, desc_kmajor(a, D, ks), desc_kmajor(bak, C + D, ks), idN192, 1);
                umma_commit(&s.barM2);
            }
        }
        ok = mbar_wait(&s.barM2, par) && ok;
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0 && chunk + 1 < cl) { issue_B(chunk + 1); ++b_issued; }

        // o = scale * O, staged as bf16 rows
        {
            const int c0 = 32 * half;
            float r[32];
            tmem_ld32(tOT + lane_base + c0, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) ost[(c0 + j) * D + v] = f2bf(scale * r[j]);
        }
        fence_async_smem();
        o_t0 = ci.t0;
        o_L = ci.L;
    }
    __syncthreads();
    if (ok) store_o_rows();
    if (o_thread) bulk_wait_all();
    if (!ok) raise_status(ws, KDA_ERR_TIMEOUT);

    // final state
    if (ok && hT) {
        for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
            float r[32];
            tmem_ld32(tS + lane_base + c0, r);
#pragma unroll
            for (int j = 0; j < 32; j += 4)   // a row per lane: 16-byte stores
                *reinterpret_cast<float4*>(hT + sidx + (size_t)v * D + c0 + j) = make_float4(r[j], r[j + 1], r[j + 2], r[j + 3]);
        }
    }
    if (tid == 0) {
        // drain copies still in flight (only after an aborted scan), bounded
        for (; a_done < a_issued; ++a_done) mbar_wait(&s.barA[a_done & 1], (uint32_t)((a_done >> 1) & 1));
        for (; b_done < b_issued; ++b_done) mbar_wait(&s.barB, (uint32_t)(b_done & 1));
        bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
    // the last CTA of the scan to finish marks the forward complete, unless a kernel of the
    // forward raised an error (the backward checks this word)
    if (tid == 0) {
        __threadfence();
        const unsigned total = gridDim.x * gridDim.y;
        if (atomicAdd(reinterpret_cast<unsigned*>(ws + kFwdCountOff), 1u) == total - 1u) {
            __threadfence();
            if (read_status(ws) == 0) *reinterpret_cast<volatile uint32_t*>(ws + kStampDoneOff) = kFwdDone;
        }
    }
}

}  // namespace kda
