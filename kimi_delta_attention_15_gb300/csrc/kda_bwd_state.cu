// Backward, state-side products of each chunk, all chunks in parallel. From the
// checkpoints S0^T (forward) and dS_L^T (backward scan), stored key-major by the
// scans, and Ut, dUt, dO of the chunk, with tcgen05 tf32 MMAs (M = 128 over the
// key channel k):
//   dQbar = scale dO S0            [c][k]
//   dW    = -dUt S0                [c][k], stored as K-major panels (umma.cuh) for the
//                                  tcgen05 products of the WY kernel
//   dKbar = Ut dS_L                [c][k]
//   dAqk  = scale dO Ut^T          [i][j], kept for j <= i
//   dgam  = sum_v dS_L[v,k] S0[v,k]  (adjoint of exp(G_L) through the decayed state,
//                                    before the factor exp(G_L))
// These are the reverse mode of Ut = U - W S0^T, O = scale[(Q^*Gamma) S0^T + Aqk Ut],
// S_L = S0 diag(exp(G_L)) + Ut^T (K^*e^{G_L-G}).
//
// Persistent and warp-specialised. Every product contracts over the value
// channel v, so a tile streams through shared memory as four 32-column value
// panels, in two rings: the S0^T and dS_L^T panels (two thirds of the bytes) in
// two stages, Ut, dUt and their split parts in three. A stage of the second ring stays in
// use from its copy through the split to the end of the MMAs that read it, the longest
// hold, so that ring gets the third stage (three stages for the first ring and two for
// the second: 0.856 ms at T=8192, H=96; the other way round: 0.762 ms):
//   warp 0        bulk copies of the panels: lane 0 the S0^T / dS_L^T ring (two stages),
//                 lane 1 the Ut / dUt ring (three stages: a stage is held from its copy
//                 through the split to the end of its MMAs) and, one tile ahead, the next
//                 tile's dO rows
//   warps 2..7    split Ut, dUt into tf32 high + low parts and dO to fp32 and hand them to
//                 the MMAs; then warps 4..7 sum the diagonal dgam on the CUDA cores (a stage of
//                 the S0^T / dS_L^T ring is free once the MMAs and these warps are done with it)
//   warp 1        the MMAs of a panel into one of two TMEM accumulator sets
//   warps 8..15   accumulators -> workspace, overlapping the next tile's MMAs
// S0, dS_L and dO are exact in tf32; Ut and dUt enter as high + low parts.
#include "kda_internal.cuh"
#include "umma.cuh"

namespace kda {

namespace {
constexpr int kStWarps = 16;
constexpr uint32_t kPanelDD = D * 128;   // one 32-column panel of a 128-row tile (16 KB)
constexpr uint32_t kPanelCD = C * 128;   // one 32-column panel of a 64-row tile (8 KB)
constexpr int kDoPitch = 2 * D + 64;     // bytes per staged dO row (padded against bank conflicts)

constexpr int kStA = 2, kStB = 3;        // stages of the two rings
constexpr int kSplitThreads = 192;       // warps 2..7 split the operands; warps 4..7 also sum dgam
struct StageA {
    uint8_t S0T[kPanelDD];   // S0^T   [128 k][32 v]
    uint8_t DST[kPanelDD];   // dS_L^T [128 k][32 v]
};
struct StageB {
    uint8_t STK[kPanelDD];   // rows 0..63 dO [c][32 v] (fp32), rows 64..127 dUt high part
    uint8_t DUL[kPanelCD];   // dUt low part [64 c][32 v]
    uint8_t UH[kPanelCD];    // Ut as copied, then its high part [64 c][32 v]
    uint8_t UL[kPanelCD];    // Ut low part
};
struct BStateSmem {
    StageA sa[kStA];
    StageB sb[kStB];
    uint8_t dos[2][C * kDoPitch];   // dO rows of a tile as stored (bf16), by tile parity
    uint64_t fullA[kStA], emptyA[kStA], fullB[kStB], emptyB[kStB], ready[kStB], tfull[2], tempty[2], fin;
    uint64_t dfull[2];              // dO rows of a tile landed, by tile parity
    uint32_t tmem;
    int abort;
};
static_assert(sizeof(BStateSmem) + 1024 <= 227 * 1024, "shared memory");
}  // namespace

size_t bwd_state_smem_bytes() { return sizeof(BStateSmem) + 1024; }

__global__ void __launch_bounds__(kStWarps * 32, 1)
    kda_bwd_state_kernel(const uint16_t* __restrict__ dO, int H, float scale, uint8_t* __restrict__ ws, Layout lay) {
    extern __shared__ uint8_t smem_raw[];
    BStateSmem& s = *reinterpret_cast<BStateSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (read_status(ws) != 0) return;
    const ChunkInfo* chunks = reinterpret_cast<const ChunkInfo*>(ws + lay.chunks);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = lay.nc_max * H;

    if (warp == 0) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kStA; ++i) {
            mbar_init(&s.fullA[i], 1);
            mbar_init(&s.emptyA[i], 1 + 128);   // the MMAs' commit and the 128 splitter threads
        }
        for (int i = 0; i < kStB; ++i) {
            mbar_init(&s.fullB[i], 1);
            mbar_init(&s.emptyB[i], 1);
            mbar_init(&s.ready[i], kSplitThreads);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], 1);
            mbar_init(&s.tempty[i], 256);
            mbar_init(&s.dfull[i], 1);
        }
        mbar_init(&s.fin, 1);
        s.abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s.tmem;
    volatile int* abort_flag = &s.abort;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // lane 0: the S0^T / dS_L^T ring, lane 1: the Ut / dUt ring (and the dO rows); the
        // two lanes run the same tile sequence independently
        if (lane < 2) {
            const bool ring_a = lane == 0;
            int it = 0, d_issued = 0;
            bool ok = true;
            // dO rows of tile t_i (the n-th of this CTA) into dos[n & 1], completing dfull[n & 1]
            auto issue_dO = [&](int t_i, int nn) {
                if (t_i >= ntiles) return;
                const int chunk = t_i / H, h = t_i - chunk * H;
                const ChunkInfo cn = chunks[chunk];
                if (cn.L <= 0) return;
                mbar_arrive_expect_tx(&s.dfull[nn & 1], (uint32_t)cn.L * 2 * D);
                for (int c = 0; c < cn.L; ++c)
                    bulk_g2s(s.dos[nn & 1] + c * kDoPitch, dO + ((size_t)(cn.t0 + c) * H + h) * D, 2 * D,
                             &s.dfull[nn & 1]);
                ++d_issued;
            };
            if (!ring_a) issue_dO(blockIdx.x, 0);
            for (int tile = blockIdx.x, n = 0; tile < ntiles && ok; tile += gridDim.x) {
                const int chunk = tile / H, h = tile - chunk * H;
                const ChunkInfo ci = chunks[chunk];
                if (ci.L <= 0) continue;
                const size_t t = (size_t)chunk * H + h;
                const uint8_t* gS0 = ws + lay.s0 + t * kTileDD;
                const uint8_t* gDS = ws + lay.ds + t * kTileDD;
                const uint8_t* gUt = ws + lay.ut + t * kTileCK;
                const uint8_t* gdU = ws + lay.dut + t * kTileCK;
                for (int p = 0; p < 4; ++p, ++it) {
                    if (ring_a) {
                        const int sa = it % kStA;
                        if (!mbar_wait(&s.emptyA[sa], (uint32_t)(((it / kStA) & 1) ^ 1)) || *abort_flag) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&s.fullA[sa], 2 * kPanelDD);
                        bulk_g2s(s.sa[sa].S0T, gS0 + p * kPanelDD, kPanelDD, &s.fullA[sa]);
                        bulk_g2s(s.sa[sa].DST, gDS + p * kPanelDD, kPanelDD, &s.fullA[sa]);
                    } else {
                        const int sb = it % kStB;
                        if (!mbar_wait(&s.emptyB[sb], (uint32_t)(((it / kStB) & 1) ^ 1)) || *abort_flag) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&s.fullB[sb], 2 * kPanelCD);
                        bulk_g2s(s.sb[sb].UH, gUt + p * kPanelCD, kPanelCD, &s.fullB[sb]);
                        bulk_g2s(s.sb[sb].STK + kPanelCD, gdU + p * kPanelCD, kPanelCD, &s.fullB[sb]);
                        // the next tile's dO rows: the splitter is done with the tile before this
                        // one once panel 2's stage was free (its previous use was panel 0 here)
                        if (p == 2) issue_dO(tile + (int)gridDim.x, n + 1);
                    }
                }
                ++n;
            }
            if (!ok) *abort_flag = 1;
            // copies still in flight (only after an abort): the last issue of each stage
            if (ring_a)
                for (int j = it - 1; j >= 0 && j >= it - kStA; --j) mbar_wait(&s.fullA[j % kStA], (uint32_t)((j / kStA) & 1));
            else {
                for (int j = it - 1; j >= 0 && j >= it - kStB; --j) mbar_wait(&s.fullB[j % kStB], (uint32_t)((j / kStB) & 1));
                for (int j = d_issued - 1; j >= 0 && j >= d_issued - 2; --j)
                    mbar_wait(&s.dfull[j & 1], (uint32_t)((j >> 1) & 1));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t id128 = idesc_tf32(128, 128, 0, 0), id64 = idesc_tf32(128, 64, 0, 0);
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x, n = 0; tile < ntiles && ok; tile += gridDim.x) {
                if (chunks[tile / H].L <= 0) continue;
                const int tb = n & 1;
                const uint32_t acc = tm + 256u * tb;
                for (int p = 0; p < 4; ++p, ++it) {
                    const int sa = it % kStA, sb = it % kStB;
                    // the split operands are ready and the S0^T / dS_L^T panels have landed
                    if (!mbar_wait(&s.ready[sb], (uint32_t)((it / kStB) & 1)) || !mbar_wait(&s.fullA[sa], (uint32_t)((it / kStA) & 1)) ||
                        (p == 0 && !mbar_wait(&s.tempty[tb], ((n >> 1) & 1) ^ 1)) || *abort_flag) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const StageA& ga = s.sa[sa];
                    const StageB& g = s.sb[sb];
                    const uint32_t aS = smem_u32(ga.S0T), aD = smem_u32(ga.DST), aK = smem_u32(g.STK);
                    const uint32_t bDL = smem_u32(g.DUL), bUH = smem_u32(g.UH), bUL = smem_u32(g.UL);
                    // [dQbar / scale | dUt S0]^T = S0^T [dO ; dUt]^T     -> cols 0..127
                    for (int ks = 0; ks < 4; ++ks)
                        umma_tf32(acc, desc_kmajor(aS, D, ks), desc_kmajor(aK, D, ks), id128, (p | ks) != 0);
                    for (int ks = 0; ks < 4; ++ks)
                        umma_tf32(acc + 64, desc_kmajor(aS, D, ks), desc_kmajor(bDL, C, ks), id64, 1);
                    // dKbar^T = dS_L^T Ut^T                              -> cols 128..191
                    for (int ks = 0; ks < 4; ++ks)
                        umma_tf32(acc + 128, desc_kmajor(aD, D, ks), desc_kmajor(bUH, C, ks), id64, (p | ks) != 0);
                    for (int ks = 0; ks < 4; ++ks)
                        umma_tf32(acc + 128, desc_kmajor(aD, D, ks), desc_kmajor(bUL, C, ks), id64, 1);
                    // [dO ; dUt] Ut^T (rows 0..63 used, x scale)          -> cols 192..255
                    for (int ks = 0; ks < 4; ++ks)
                        umma_tf32(acc + 192, desc_kmajor(aK, D, ks), desc_kmajor(bUH, C, ks), id64, (p | ks) != 0);
                    for (int ks = 0; ks < 4; ++ks)
                        umma_tf32(acc + 192, desc_kmajor(aK, D, ks), desc_kmajor(bUL, C, ks), id64, 1);
                    umma_commit(&s.emptyA[sa]);
                    umma_commit(&s.emptyB[sb]);
                    if (p == 3) umma_commit(&s.tfull[tb]);
                }
                ++n;
            }
            if (!ok) *abort_flag = 1;
            umma_commit(&s.fin);   // every MMA of this CTA has completed once fin flips
            mbar_wait(&s.fin, 0);
        }
        __syncwarp();
    } else if (warp >= 2 && warp < 8) {
        // --------------------------------------------------------- splitter
        const int t2 = tid - 64;    // item index of the split (0 .. 191)
        const int t = tid - 128;    // row k of the key-major panels, for dgam (warps 4..7)
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x, n = 0; tile < ntiles && ok; tile += gridDim.x) {
            const int chunk = tile / H;
            const ChunkInfo ci = chunks[chunk];
            if (ci.L <= 0) continue;
            const uint8_t* dos = s.dos[n & 1];
            float dg = 0.0f;
            for (int p = 0; p < 4; ++p, ++it) {
                const int sa = it % kStA, sg = it % kStB;
                // warp-uniform decisions: each warp's arrivals are made by one lane
                if (!__all_sync(0xffffffffu, mbar_wait(&s.fullB[sg], (uint32_t)((it / kStB) & 1)) &&
                                                 (p != 0 || mbar_wait(&s.dfull[n & 1], (uint32_t)((n >> 1) & 1))) &&
                                                 !*abort_flag)) {
                    ok = false;
                    break;
                }
                StageB& g = s.sb[sg];
                // Ut, dUt -> high (in place) + low parts; dO rows -> fp32 (zero past the chunk):
                // 512 items of 16 bytes, 192 threads
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    const int e = t2 + kSplitThreads * r, c = e >> 3, j4 = e & 7;
                    if (e >= 4 * C * 2) break;
                    const uint32_t off = c * 128u + ((j4 ^ (c & 7)) << 4);
                    float4 x = *reinterpret_cast<const float4*>(g.UH + off);
                    float4 xh = make_float4(tf32_round(x.x), tf32_round(x.y), tf32_round(x.z), tf32_round(x.w));
                    *reinterpret_cast<float4*>(g.UH + off) = xh;
                    *reinterpret_cast<float4*>(g.UL + off) =
                        make_float4(tf32_round(x.x - xh.x), tf32_round(x.y - xh.y), tf32_round(x.z - xh.z),
                                    tf32_round(x.w - xh.w));
                    x = *reinterpret_cast<const float4*>(g.STK + kPanelCD + off);
                    xh = make_float4(tf32_round(x.x), tf32_round(x.y), tf32_round(x.z), tf32_round(x.w));
                    *reinterpret_cast<float4*>(g.STK + kPanelCD + off) = xh;
                    *reinterpret_cast<float4*>(g.DUL + off) =
                        make_float4(tf32_round(x.x - xh.x), tf32_round(x.y - xh.y), tf32_round(x.z - xh.z),
                                    tf32_round(x.w - xh.w));
                    float4 d = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (c < ci.L) {
                        const uint2 w = *reinterpret_cast<const uint2*>(dos + c * kDoPitch + 2 * (32 * p + 4 * j4));
                        d = make_float4(bf2f((uint16_t)(w.x & 0xffffu)), bf2f((uint16_t)(w.x >> 16)),
                                        bf2f((uint16_t)(w.y & 0xffffu)), bf2f((uint16_t)(w.y >> 16)));
                    }
                    *reinterpret_cast<float4*>(g.STK + off) = d;
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive_cnt(&s.ready[sg], 32);
                if (t < 0) continue;   // warps 2, 3: the split only
                // dgam: row k of S0^T and dS_L^T, after the split is handed to the MMAs; the
                // stage of these panels is released by this warp's arrival (32 counts) and the MMAs' commit
                if (!__all_sync(0xffffffffu, mbar_wait(&s.fullA[sa], (uint32_t)((it / kStA) & 1)) && !*abort_flag)) {
                    ok = false;
                    break;
                }
                const StageA& ga = s.sa[sa];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const uint32_t off = t * 128u + ((j4 ^ (t & 7)) << 4);
                    const float4 a = *reinterpret_cast<const float4*>(ga.S0T + off);
                    const float4 b = *reinterpret_cast<const float4*>(ga.DST + off);
                    dg = fmaf(a.x, b.x, dg); dg = fmaf(a.y, b.y, dg);
                    dg = fmaf(a.z, b.z, dg); dg = fmaf(a.w, b.w, dg);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_cnt(&s.emptyA[sa], 32);
            }
            if (!ok) break;
            const size_t tt = (size_t)chunk * H + (tile - chunk * H);
            if (t >= 0) reinterpret_cast<float*>(ws + lay.bg + tt * BgOff::BYTES + BgOff::DGAM)[t] = dg;
            ++n;
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 8) {
        // --------------------------------------------------------- epilogue
        const int e = tid - 256, ew = e >> 5, q = ew & 3, hf = ew >> 2;
        const int kq = 32 * q + lane;   // TMEM lane: key channel k (row i for dAqk)
        bool ok = true;
        for (int tile = blockIdx.x, n = 0; tile < ntiles && ok; tile += gridDim.x) {
            const int chunk = tile / H;
            if (chunks[chunk].L <= 0) continue;
            const int tb = n & 1;
            // the TMEM loads below are warp-collective: decide per warp
            if (!__all_sync(0xffffffffu, mbar_wait(&s.tfull[tb], (n >> 1) & 1) && !*abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t acc = tm + 256u * tb + ((uint32_t)(32 * q) << 16);
            const size_t tt = (size_t)chunk * H + (tile - chunk * H);
            uint8_t* bg = ws + lay.bg + tt * BgOff::BYTES;
            float r[32];
            if (hf == 0) {
                float* gdQ = reinterpret_cast<float*>(bg + BgOff::DQB);
                tmem_ld32(acc + 0, r);
#pragma unroll
                for (int j = 0; j < 32; ++j) gdQ[j * D + kq] = scale * r[j];
                tmem_ld32(acc + 32, r);
#pragma unroll
                for (int j = 0; j < 32; ++j) gdQ[(32 + j) * D + kq] = scale * r[j];
                tmem_ld32(acc + 64, r);
#pragma unroll
                for (int j = 0; j < 32; ++j) *reinterpret_cast<float*>(bg + BgOff::DW + panel_off(j, kq, C)) = -r[j];
            } else {
                float* gdK = reinterpret_cast<float*>(bg + BgOff::DKB);
                tmem_ld32(acc + 96, r);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    *reinterpret_cast<float*>(bg + BgOff::DW + panel_off(32 + j, kq, C)) = -r[j];
                tmem_ld32(acc + 128, r);
#pragma unroll
                for (int j = 0; j < 32; ++j) gdK[j * D + kq] = r[j];
                tmem_ld32(acc + 160, r);
#pragma unroll
                for (int j = 0; j < 32; ++j) gdK[(32 + j) * D + kq] = r[j];
            }
            if (q < 2) {
                float* gdA = reinterpret_cast<float*>(bg + BgOff::DAQK);
                const int i = kq, j0 = 32 * hf;
                tmem_ld32(acc + 192 + j0, r);
                // a row per lane: 16-byte stores (a warp store covers 32 rows)
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float a4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) a4[e] = (j0 + j + e <= i) ? scale * r[j + e] : 0.0f;
                    *reinterpret_cast<float4*>(gdA + i * C + j0 + j) = make_float4(a4[0], a4[1], a4[2], a4[3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cnt(&s.tempty[tb], 32);
            ++n;
        }
        if (!ok) *abort_flag = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && tid == 0) raise_status(ws, KDA_ERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

}  // namespace kda
