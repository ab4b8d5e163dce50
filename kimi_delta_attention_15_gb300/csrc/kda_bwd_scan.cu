// Backward state scan: one CTA per (sequence, head), chunks in reverse order.
// The fp32 state adjoint dS (V x K) lives in tensor memory. Per chunk, given
// dS_L (adjoint of the chunk's final state):
//   dUt^T = scale dO^T Aqk + dS_L (K^*e^{G_L-G})^T             (tcgen05, M=128 N=64)
//   dS_0  = dS_L diag(exp(G_L)) + scale dO^T (Q^*Gamma) - dUt^T W
// which is the reverse mode of the chunk form
//   Ut = U - W S0^T,  O = scale[(Q^*Gamma) S0^T + Aqk Ut],
//   S_L = S0 diag(exp(G_L)) + Ut^T (K^*e^{G_L-G}).
// dS_L^T of every chunk (tf32, as the MMAs use it) and dUt (fp32) are stored in the
// workspace for the per-chunk backward kernels; dh0 = dS at the sequence start.
// dS_L enters the MMA from a tf32 copy in tensor memory (A operand in TMEM). The
// two products with A = dO^T run as one MMA over stacked B operands:
//   dUt^T = dS_L KB^T;  [dUt^T | dS] += dO^T [scale Aqk ; Q^*Gamma]      (N = 192)
// so TMEM holds dUt^T (columns 0..63), dS (64..191), tf32 dS_L (256..383). W^T, used
// by the second MMA only, is double-buffered and requested two chunks ahead.
#include "kda_internal.cuh"
#include "umma.cuh"

namespace kda {

namespace {
struct BScanSmem {
    uint8_t WT[2][kTileCK];  // W^T [128 k][64 c]: bulk group Y (second MMA), by chunk parity
    // [Aqk^T ; QB^T] as one 192-row operand: panel p = Aqk^T rows (8 KB) then QB^T rows (16 KB)
    uint8_t AQ[kTileCK + kTileCC];   // \ bulk group X (first MMA)
    uint8_t KB[kTileCK];             // / KB [64 c][128 k]
    uint8_t DOT[kTileCK];    // dO^T [128 v][64 i], then -dUt^T [128 v][64 c]
    uint16_t DO[C * D];      // dO rows of the next chunk as stored (bf16 [64 i][128 v]), cp.async
    float gam[D];
    uint64_t barX, barY[2], barM1, barM2;
    uint32_t tmem;
};
}  // namespace

size_t bwd_scan_smem_bytes() { return sizeof(BScanSmem) + 1024; }

__global__ void __launch_bounds__(256, 1)
    kda_bwd_scan_kernel(const uint16_t* __restrict__ dO, const float* __restrict__ dhT, float* __restrict__ dh0,
                        int H, uint8_t* __restrict__ ws, Layout lay, uint64_t shape_hash) {
    extern __shared__ uint8_t smem_raw[];
    BScanSmem& s = *reinterpret_cast<BScanSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (read_status(ws) != 0) return;
    // the workspace must hold a completed forward of this shape (its provenance stamp);
    // every CTA reads the same words, so all of them return or none
    if (*reinterpret_cast<const volatile uint64_t*>(ws + kStampHashOff) != shape_hash ||
        *reinterpret_cast<const volatile uint32_t*>(ws + kStampDoneOff) != kFwdDone) {
        if (threadIdx.x == 0) raise_status(ws, KDA_ERR_STALE_WORKSPACE);
        return;
    }
    const int h = blockIdx.x;
    const int n = reinterpret_cast<const int*>(ws + lay.seq_order)[blockIdx.y];
    const int cf = reinterpret_cast<const int*>(ws + lay.seq_first)[n];
    const int cl = reinterpret_cast<const int*>(ws + lay.seq_first)[n + 1];
    const ChunkInfo* chunks = reinterpret_cast<const ChunkInfo*>(ws + lay.chunks);
    const int tid = threadIdx.x, warp = tid >> 5;
    // threads v and v + 128 own adjoint row v (TMEM lane v) and split its columns
    const int v = tid & (D - 1), half = tid >> 7;
    const size_t sidx = ((size_t)n * H + h) * D * D;

    if (warp == 0) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&s.barX, 1); mbar_init(&s.barY[0], 1); mbar_init(&s.barY[1], 1); mbar_init(&s.barM1, 1); mbar_init(&s.barM2, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s.tmem;
    const uint32_t tU = tm, tS = tm + 64, tDS = tm + 256;   // tDS: tf32 copy of dS_L
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
        float r[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {   // a row per lane: 16-byte loads
            const float4 x = dhT ? *reinterpret_cast<const float4*>(dhT + sidx + (size_t)v * D + c0 + j)
                                 : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            r[j] = x.x; r[j + 1] = x.y; r[j + 2] = x.z; r[j + 3] = x.w;
        }
        tmem_st32(tS + lane_base + c0, r);
    }

    auto img_of = [&](int chunk) { return ws + lay.img + ((size_t)chunk * H + h) * ImgOff::BYTES; };
    auto issue_X = [&](int chunk) {
        const uint8_t* img = img_of(chunk);
        mbar_arrive_expect_tx(&s.barX, (uint32_t)(2 * kTileCK + kTileCC));
        for (int p = 0; p < 2; ++p) {
            bulk_g2s(s.AQ + p * (C + D) * 128, img + ImgOff::AQKT + p * C * 128, C * 128, &s.barX);
            bulk_g2s(s.AQ + p * (C + D) * 128 + C * 128, img + ImgOff::QBT + p * D * 128, D * 128, &s.barX);
        }
        bulk_g2s(s.KB, img + ImgOff::KB, (uint32_t)kTileCK, &s.barX);
    };
    // W^T of the i-th chunk from the end goes to buffer i & 1, phase (i >> 1) of barY[i & 1]
    auto issue_Y = [&](int chunk) {
        const int b = (cl - 1 - chunk) & 1;
        mbar_arrive_expect_tx(&s.barY[b], (uint32_t)kTileCK);
        bulk_g2s(s.WT[b], img_of(chunk) + ImgOff::WT, (uint32_t)kTileCK, &s.barY[b]);
    };
    int x_issued = 0, y_issued = 0, x_done = 0, y_done = 0;   // in chunk order (thread 0)
    if (tid == 0 && cf < cl) {
        issue_X(cl - 1);
        issue_Y(cl - 1);
        x_issued = y_issued = 1;
        if (cl - 2 >= cf) { issue_Y(cl - 2); y_issued = 2; }
    }

    bool ok = true;
    const uint32_t idN64 = idesc_tf32(128, 64, 0, 0);
    const uint32_t idN128 = idesc_tf32(128, 128, 0, 0);
    const uint32_t idN192 = idesc_tf32(128, 192, 0, 0);
    // dO rows of a chunk -> s.DO (rows past the chunk's end read as zero); 16 bytes per
    // copy, four copies per thread, issued one chunk ahead of use
    auto issue_dO = [&](const ChunkInfo& c2) {
#pragma unroll
        for (int r = 0; r < (C * D / 8) / 256; ++r) {
            const int seg = tid + 256 * r, i = seg >> 4, c8 = (seg & 15) * 8;
            const bool valid = i < c2.L;
            const uint16_t* src = dO + ((size_t)(c2.t0 + (valid ? i : 0)) * H + h) * D + c8;
            cp_async16_zfill(s.DO + i * D + c8, src, valid);
        }
        cp_async_commit();
    };
    // exp(G_L) and the chunk record are read one chunk ahead
    float gam_next = cf < cl ? reinterpret_cast<const float*>(img_of(cl - 1) + ImgOff::GAML)[v] : 0.0f;
    if (cf < cl) issue_dO(chunks[cl - 1]);
    for (int chunk = cl - 1; chunk >= cf && ok; --chunk) {
        const uint32_t par = (uint32_t)((cl - 1 - chunk) & 1);
        const size_t tile = (size_t)chunk * H + h;
        if (half == 0) s.gam[v] = gam_next;
        ChunkInfo ci_prev{0, 0, 0, 0};
        if (chunk - 1 >= cf) {
            ci_prev = chunks[chunk - 1];
            gam_next = reinterpret_cast<const float*>(img_of(chunk - 1) + ImgOff::GAML)[v];
        }
        cp_async_wait_all();
        __syncthreads();
        // dO^T into the operand tile (row v, columns i); bf16 values are exact in tf32
        // (the output scale is folded into the Aqk^T and (Q^*Gamma)^T images)
#pragma unroll
        for (int ii = 0; ii < C / 2; ii += 4) {
            const uint16_t* col = s.DO + (32 * half + ii) * D + v;
            *reinterpret_cast<float4*>(s.DOT + panel_off(v, 32 * half + ii, D)) =
                make_float4(bf2f(col[0]), bf2f(col[D]), bf2f(col[2 * D]), bf2f(col[3 * D]));
        }
        // dS_L: TMEM -> tf32 copy in TMEM (the MMA operand); dS_L diag(exp(G_L)) back to TMEM
        // (both 32-column halves in flight at once: one wait for the loads, one for the stores).
        // The checkpoint dS_L^T [k][v] is written from the tf32 copy once the MMAs run.
        uint8_t* gDST = ws + lay.ds + tile * kTileDD;
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
            tmem_st32_issue(tDS + lane_base + cb, q0);
            tmem_st32_issue(tDS + lane_base + cb + 32, q1);
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
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (chunk - 1 >= cf) issue_dO(ci_prev);   // every thread is past its reads of s.DO
        if (tid == 0) {
            if (!mbar_wait(&s.barX, par)) ok = false;
            else ++x_done;
            if (ok) {
                // dUt^T = dS_L KB^T
                for (int ks = 0; ks < D / 8; ++ks)
                    umma_tf32_ta(tU, tDS + 8 * ks, desc_kmajor(smem_u32(s.KB), C, ks), idN64, ks > 0);
                // [dUt^T | dS] += dO^T [scale Aqk ; scale QB]
                for (int ks = 0; ks < C / 8; ++ks)
                    umma_tf32(tU, desc_kmajor(smem_u32(s.DOT), D, ks), desc_kmajor(smem_u32(s.AQ), C + D, ks),
                              idN192, 1);
                umma_commit(&s.barM1);
            }
        }
        // the checkpoint dS_L^T, read back from its tf32 copy while the MMAs read the same copy
        {
            const int cb = 64 * half;
            uint32_t q0[32], q1[32];
            tmem_ld32_issue(tDS + lane_base + cb, q0);
            tmem_ld32_issue(tDS + lane_base + cb + 32, q1);
            tmem_wait_ld(q0);
            tmem_after_wait(q1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                *reinterpret_cast<uint32_t*>(gDST + panel_off(cb + j, v, D)) = q0[j];
                *reinterpret_cast<uint32_t*>(gDST + panel_off(cb + 32 + j, v, D)) = q1[j];
            }
        }
        ok = mbar_wait(&s.barM1, par) && ok;
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0 && chunk - 1 >= cf) { issue_X(chunk - 1); ++x_issued; }

        // -dUt^T into the operand tile (reusing DOT); dUt (fp32) -> workspace [c][v] panels
        uint8_t* gdU = ws + lay.dut + tile * kTileCK;
        float du[32];   // to the workspace once the state update is issued
        {
            const int c0 = 32 * half;
            tmem_ld32(tU + lane_base + c0, du);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(s.DOT + panel_off(v, c0 + j, D)) = make_float4(
                    -tf32_round(du[j]), -tf32_round(du[j + 1]), -tf32_round(du[j + 2]), -tf32_round(du[j + 3]));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const int yb = (cl - 1 - chunk) & 1;
        if (tid == 0) {
            if (!mbar_wait(&s.barY[yb], (uint32_t)(((cl - 1 - chunk) >> 1) & 1))) ok = false;
            else ++y_done;
            if (ok) {
                for (int ks = 0; ks < C / 8; ++ks)
                    umma_tf32(tS, desc_kmajor(smem_u32(s.DOT), D, ks), desc_kmajor(smem_u32(s.WT[yb]), D, ks),
                              idN128, 1);
                umma_commit(&s.barM2);
            }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) *reinterpret_cast<float*>(gdU + panel_off(32 * half + j, v, C)) = du[j];
        ok = mbar_wait(&s.barM2, par) && ok;
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        if (tid == 0 && chunk - 2 >= cf) { issue_Y(chunk - 2); ++y_issued; }   // into this chunk's buffer
    }
    if (!ok) raise_status(ws, KDA_ERR_TIMEOUT);
    if (ok && dh0) {
        for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
            float r[32];
            tmem_ld32(tS + lane_base + c0, r);
#pragma unroll
            for (int j = 0; j < 32; j += 4)   // a row per lane: 16-byte stores
                *reinterpret_cast<float4*>(dh0 + sidx + (size_t)v * D + c0 + j) = make_float4(r[j], r[j + 1], r[j + 2], r[j + 3]);
        }
    }
    if (tid == 0) {
        for (; x_done < x_issued; ++x_done) mbar_wait(&s.barX, (uint32_t)(x_done & 1));
        for (; y_done < y_issued; ++y_done) mbar_wait(&s.barY[y_done & 1], (uint32_t)((y_done >> 1) & 1));
        bulk_wait_all();
    }
    cp_async_wait_all();   // dO copies still in flight (only after an aborted scan)
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace kda
