// Backward through the UT transform of each chunk, on tcgen05: persistent CTAs (one
// per SM) over all (chunk, head) tiles. With W = T (K^*Gamma), U = T V,
// T = X diag(beta), X = (I + A)^{-1}, A = diag(beta) B, and the adjoints dW
// (state-products kernel) and dU = dUt (backward scan):
//   dT    = dW (K^*Gamma)^T + dU V^T
//   dKt   = T^T dW        (adjoint of K^*Gamma)
//   dV    = T^T dU        (final dv)
//   dbeta_j  = sum_i dT_ij X_ij + sum_l dA_jl B_jl
//   dA    = -strict_lower(X^T dT T^T),   dB = diag(beta) dA
// (the reverse mode of the "16-sub-chunk + WY" chunk form of the kda-neuron-kernels log).
//
// Every product is a dense tcgen05 kind::tf32 MMA with an fp32 accumulator in tensor
// memory; operands are K-major panels (umma.cuh) in shared memory. Single tf32
// products: the measured output errors against the fp64 reference stay well inside
// their tolerances (the pair-term kernel is the one that needs split operands).
// tf32 operands are K-major only, so the products that contract over the chunk rows
// read transposed copies, made in shared memory:
//   1. dT            = [dW | dU] [K~ | V]^T          (M = 64,  N = 64, K = 256)
//   2. [dKt^T; dV^T] = [dW^T ; dU^T] T               (M = 128 twice, N = 64, K = 64)
//   3. M^T           = T dT^T                        (M = 64, N = 64, K = 64), M = dT T^T
//   4. dA'           = X^T M                         (M = 64, N = 64, K = 64)
// Products 2 and 3 run back to back; 4 waits for the readback of 3.
//
// K~ = K^*Gamma comes from the forward's images (so this kernel prepares no rows), as do
// X and B. dW, dU, K~, X and B arrive by bulk copy and the raw v rows by cp.async, each
// issued during the previous tile as soon as its buffer is free. The kernel writes dKt
// (fp32), dv (bf16), dB (fp32) and dbeta.
#include "kda_internal.cuh"
#include "umma.cuh"

namespace kda {

namespace {
constexpr int kWyWarps = 16;
constexpr int kWyThreads = kWyWarps * 32;
// issues every tcgen05 product (an MMA issue takes tens of cycles, and the rest of its warp
// waits meanwhile: the last warp has the least other work)
constexpr int kMmaThread = (kWyWarps - 1) * 32;
// row pitch of the staged raw v rows (bf16): 272 bytes, so that eight consecutive rows
// read at one column hit eight different 16-byte bank groups
constexpr int kVsPitch = D + 8;

struct WySmem {
    // operand tiles, 1024-byte aligned (umma.cuh panels)
    uint8_t dW[kTileCK];       // dW [64 i][128 c] (bulk copy)
    uint8_t dU[kTileCK];       // dU [64 i][128 v] (bulk copy)
    uint8_t KV[2 * kTileCK];   // K~ [64 j][128 c] (bulk copy) | V [64 j][128 v] (from the raw
                               // rows, staged bf16 at a 272-byte pitch in its first 17 KB); after product 1 the
                               // stacked [dW^T ; dU^T] [256][64 i]
    uint8_t XT[kTileCC];       // X^T [64 i][64 m]
    uint8_t TT[kTileCC];       // T^T [64 j][64 i]
    uint8_t TN[kTileCC];       // T   [64 m][64 j]
    uint8_t DT[kTileCC];       // dT  [64 i][64 j]; after product 3, M as [64 j][64 m]
    float X[C * C];            // X row-major (bulk copy)
    float Bm[C * C];           // B row-major (bulk copy)
    float beta[C];
    float dbeta[4][C];         // partial sums of dT_ij X_ij over the rows i = p mod 4
    float db2[C];              // sum_j dA_ij B_ij
    uint64_t barW, barU, barK, barX, barB, barM[4], barFin;
    uint32_t tmem;
};
static_assert(sizeof(WySmem) + 1024 <= 227 * 1024, "shared memory");

// TMEM columns of the accumulators. M = 64 products: row m in lane 32 (m / 16) + m % 16.
constexpr uint32_t kD1 = 0, kD2K = 64, kD2V = 128, kD3 = 192, kD4 = 256;
}  // namespace

size_t bwd_wy_smem_bytes() { return sizeof(WySmem) + 1024; }

// kGrouped: k holds H / G heads (grouped value heads). This kernel reads no q or k rows
// (K~ comes from the forward's images), so both instantiations run the same code; the
// template keeps the launch interface of the other chunk kernels.
template <bool kGrouped>
__global__ void __launch_bounds__(kWyThreads, 1)
    kda_bwd_wy_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                      const uint16_t* __restrict__ g_raw, const uint16_t* __restrict__ beta_raw,
                      const float* __restrict__ A_log, const float* __restrict__ dt_bias, int H, float lb,
                      uint16_t* __restrict__ dv, uint8_t* __restrict__ ws, Layout lay) {
    (void)k; (void)g_raw; (void)A_log; (void)dt_bias; (void)lb;
    extern __shared__ uint8_t smem_raw[];
    WySmem& s = *reinterpret_cast<WySmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (read_status(ws) != 0) return;
    const ChunkInfo* chunks = reinterpret_cast<const ChunkInfo*>(ws + lay.chunks);
    const int ntiles = (int)lay.nc_max * H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Persistent over tiles (tile = chunk * H + h). Empty chunk records only
    // follow the last real chunk, so the first empty tile ends the CTA's work.
    const int step = (int)gridDim.x;
    int tile_i = blockIdx.x;
    ChunkInfo ci = tile_i < ntiles ? chunks[tile_i / H] : ChunkInfo{0, 0, 0, 0};
    if (ci.L <= 0) return;

    if (warp == 0) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&s.barW, 1); mbar_init(&s.barU, 1); mbar_init(&s.barK, 1);
        mbar_init(&s.barX, 1); mbar_init(&s.barB, 1);
        for (int i = 0; i < 4; ++i) mbar_init(&s.barM[i], 1);
        mbar_init(&s.barFin, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s.tmem;
    uint16_t* const stv = reinterpret_cast<uint16_t*>(s.KV + kTileCK);   // staged raw v rows

    // bulk copies of tile t_i into one buffer each, completing a phase of the barrier
    auto bulk = [&](uint64_t* bar, void* dst, const uint8_t* src, uint32_t bytes) {
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(dst, src, bytes, bar);
    };
    auto img_of = [&](int t_i) { return ws + lay.img + (size_t)t_i * ImgOff::BYTES; };
    auto issue_dW = [&](int t_i) { bulk(&s.barW, s.dW, ws + lay.bg + (size_t)t_i * BgOff::BYTES + BgOff::DW, kTileCK); };
    auto issue_dU = [&](int t_i) { bulk(&s.barU, s.dU, ws + lay.dut + (size_t)t_i * kTileCK, kTileCK); };
    auto issue_K = [&](int t_i) { bulk(&s.barK, s.KV, img_of(t_i) + ImgOff::KT, kTileCK); };
    auto issue_X = [&](int t_i) { bulk(&s.barX, s.X, img_of(t_i) + ImgOff::XM, kTileCC); };
    auto issue_B = [&](int t_i) { bulk(&s.barB, s.Bm, img_of(t_i) + ImgOff::BM, kTileCC); };
    // raw v rows of tile t_i (record cn); rows past the chunk read as zero; beta_raw
    uint16_t braw_next = 0;
    auto stage_v = [&](int t_i, const ChunkInfo& cn) {
        const int hn = t_i % H;
        if (tid < C) braw_next = tid < cn.L ? beta_raw[(size_t)(cn.t0 + tid) * H + hn] : (uint16_t)0;
        for (int seg = tid; seg < C * (D / 8); seg += kWyThreads) {
            const int r = seg >> 4, c8 = (seg & 15) * 8;
            const bool valid = r < cn.L;
            cp_async16_zfill(stv + r * kVsPitch + c8, v + ((size_t)(cn.t0 + (valid ? r : 0)) * H + hn) * D + c8, valid);
        }
        cp_async_commit();
    };

    // phases issued on each bulk barrier (thread 0: W, U, K, X, B), for the drain at the end
    int nb[5] = {0, 0, 0, 0, 0};
    if (tid == 0) {
        issue_dW(tile_i); issue_dU(tile_i); issue_K(tile_i); issue_X(tile_i); issue_B(tile_i);
        for (int i = 0; i < 5; ++i) nb[i] = 1;
    }
    stage_v(tile_i, ci);
    uint16_t braw = braw_next;
    const uint32_t id64 = idesc_tf32(64, 64, 0, 0), id128 = idesc_tf32(128, 64, 0, 0);
    const int q4 = warp & 3;                 // TMEM lane quarter of this warp
    const bool lrow = lane < 16;             // M = 64: lanes 0..15 of a quarter hold rows
    const int mrow = 16 * q4 + lane;         // the chunk row those lanes hold
    bool ok = true;
    uint32_t par = 0;
    while (true) {
        const int nxt = tile_i + step;
        const ChunkInfo cn = nxt < ntiles ? chunks[nxt / H] : ChunkInfo{0, 0, 0, 0};
        const int h = tile_i % H;
        const int L = ci.L;
        const size_t tile = (size_t)tile_i;
        uint8_t* wy = ws + lay.wy + tile * WyOff::BYTES;

        // ---- v rows -> fp32 operand V [j][v]; beta
        cp_async_wait_all();
        __syncthreads();
        {
            // thread: row r, columns c0 .. c0 + 15; consecutive lanes take consecutive rows, so
            // the panel stores below (16-byte chunk j ^ (r & 7)) are free of bank conflicts
            const int r = tid & (C - 1), c0 = (tid >> 6) * 16;
            const uint4 v0 = *reinterpret_cast<const uint4*>(stv + r * kVsPitch + c0);
            const uint4 v1 = *reinterpret_cast<const uint4*>(stv + r * kVsPitch + c0 + 8);
            if (tid < C) s.beta[tid] = tid < L ? sigmoidf(bf2f(braw)) : 0.0f;
            __syncthreads();   // every staged row is in registers: V overwrites the staging
            const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            uint8_t* V = s.KV + kTileCK;
#pragma unroll
            for (int e = 0; e < 4; ++e)   // bf16 v is exact in tf32: its fp32 bit pattern
                *reinterpret_cast<uint4*>(V + panel_off(r, c0 + 4 * e, C)) =
                    make_uint4(w[2 * e] << 16, w[2 * e] & 0xffff0000u, w[2 * e + 1] << 16, w[2 * e + 1] & 0xffff0000u);
        }
        // V and beta are in place: product 1 is issued first and the T panels are built beside it
        fence_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        // ---- product 1: dT = dW K~^T + dU V^T
        if (tid == kMmaThread) {
            if (mbar_wait(&s.barW, par) && mbar_wait(&s.barU, par) && mbar_wait(&s.barK, par)) {
                const uint32_t aW = smem_u32(s.dW), aU = smem_u32(s.dU), bK = smem_u32(s.KV),
                               bV = smem_u32(s.KV + kTileCK);
                for (int ks = 0; ks < D / 8; ++ks)
                    umma_tf32(tm + kD1, desc_kmajor(aW, C, ks), desc_kmajor(bK, C, ks), id64, ks > 0);
                for (int ks = 0; ks < D / 8; ++ks)
                    umma_tf32(tm + kD1, desc_kmajor(aU, C, ks), desc_kmajor(bV, C, ks), id64, 1);
                umma_commit(&s.barM[0]);
            } else {
                ok = false;
            }
        }
        // ---- T [m][j] = X diag(beta); X^T [i][m] and T^T = diag(beta) X^T by strips: thread
        // (row r of the transposed tile, four columns from i0) reads four rows of X. Warps 0..14,
        // while product 1 runs (the MMA thread's warp stays out)
        ok = mbar_wait(&s.barX, par) && ok;
        for (int e = tid; e < C * C / 4 && tid < kMmaThread; e += kMmaThread) {
            {   // T: 4 consecutive columns of one row
                const int m = e >> 4, j = (e & 15) * 4;
                const float4 x = *reinterpret_cast<const float4*>(s.X + m * C + j);
                const float4 b = *reinterpret_cast<const float4*>(s.beta + j);
                *reinterpret_cast<float4*>(s.TN + panel_off(m, j, C)) =
                    make_float4(tf32_round(x.x * b.x), tf32_round(x.y * b.y), tf32_round(x.z * b.z), tf32_round(x.w * b.w));
            }
            const int r = e & (C - 1), i0 = 4 * (e >> 6);
            const float x0 = s.X[(i0 + 0) * C + r], x1 = s.X[(i0 + 1) * C + r];
            const float x2 = s.X[(i0 + 2) * C + r], x3 = s.X[(i0 + 3) * C + r];
            const float br = s.beta[r];
            *reinterpret_cast<float4*>(s.XT + panel_off(r, i0, C)) =
                make_float4(tf32_round(x0), tf32_round(x1), tf32_round(x2), tf32_round(x3));
            *reinterpret_cast<float4*>(s.TT + panel_off(r, i0, C)) =
                make_float4(tf32_round(x0 * br), tf32_round(x1 * br), tf32_round(x2 * br), tf32_round(x3 * br));
        }
        fence_async_smem();
        ok = ok && mbar_wait(&s.barM[0], par);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        // ---- dT -> operand [i][j] (warps 0..7); [dW^T ; dU^T] -> stacked operand (all warps
        // afterwards: thread (row r of dW^T or dU^T, four columns from i0) reads four rows)
        if (warp < 8) {
            const int hcol = warp >> 2;
            uint32_t r[32];
            tmem_ld32_issue(tm + kD1 + ((uint32_t)(32 * q4) << 16) + 32 * hcol, r);
            tmem_wait_ld(r);
            if (lrow) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(s.DT + panel_off(mrow, 32 * hcol + j, C)) =
                        make_float4(tf32_round(__uint_as_float(r[j])), tf32_round(__uint_as_float(r[j + 1])),
                                    tf32_round(__uint_as_float(r[j + 2])), tf32_round(__uint_as_float(r[j + 3])));
            }
        }
        for (int e = tid; e < 2 * D * C / 4; e += kWyThreads) {
            const int rr = e & (2 * D - 1), i0 = 4 * (e >> 8);   // stacked row rr, columns i0 .. i0 + 3
            const uint8_t* src = rr < D ? s.dW : s.dU;
            const int c = rr & (D - 1);
            float x[4];
#pragma unroll
            for (int f = 0; f < 4; ++f) x[f] = *reinterpret_cast<const float*>(src + panel_off(i0 + f, c, C));
            *reinterpret_cast<float4*>(s.KV + panel_off(rr, i0, 2 * D)) =
                make_float4(tf32_round(x[0]), tf32_round(x[1]), tf32_round(x[2]), tf32_round(x[3]));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- products 2 and 3; dW and dU are no longer read: the next tile's stream in
        if (tid == kMmaThread) {
            const uint32_t aS = smem_u32(s.KV), bTT = smem_u32(s.TT), aTN = smem_u32(s.TN), bDT = smem_u32(s.DT);
            for (int ks = 0; ks < C / 8; ++ks)
                umma_tf32(tm + kD2K, desc_kmajor(aS, 2 * D, ks, 0), desc_kmajor(bTT, C, ks), id128, ks > 0);
            for (int ks = 0; ks < C / 8; ++ks)
                umma_tf32(tm + kD2V, desc_kmajor(aS, 2 * D, ks, D), desc_kmajor(bTT, C, ks), id128, ks > 0);
            umma_commit(&s.barM[1]);
            for (int ks = 0; ks < C / 8; ++ks)
                umma_tf32(tm + kD3, desc_kmajor(aTN, C, ks), desc_kmajor(bDT, C, ks), id64, ks > 0);
            umma_commit(&s.barM[2]);
        }
        if (tid == 0 && cn.L > 0) { issue_dW(nxt); issue_dU(nxt); ++nb[0]; ++nb[1]; }
        // dbeta_j = sum_{i >= j} dT_ij X_ij: warps 0..7, thread (column j = lane-consecutive,
        // rows i = p mod 4), so that a warp reads 32 consecutive columns of one row; the four
        // partial sums are combined in a fixed order at the end of the tile
        if (warp < 8) {
            const int j = tid & (C - 1), p = tid >> 6;
            float acc = 0.0f;
#pragma unroll
            for (int i = p; i < C; i += 4)
                if (i >= j) acc += *reinterpret_cast<const float*>(s.DT + panel_off(i, j, C)) * s.X[i * C + j];
            s.dbeta[p][j] = acc;
        }
        ok = ok && mbar_wait(&s.barM[2], par);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        // X is read for the last time above: the next tile's X streams in
        if (tid == 0 && cn.L > 0) { issue_X(nxt); ++nb[3]; }
        // ---- M rows -> operand [j][m] of product 4, over dT (read by product 3, complete)
        if (warp < 8) {
            const int hcol = warp >> 2;
            uint32_t r[32];
            tmem_ld32_issue(tm + kD3 + ((uint32_t)(32 * q4) << 16) + 32 * hcol, r);
            tmem_wait_ld(r);
            if (lrow) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(s.DT + panel_off(mrow, 32 * hcol + j, C)) =
                        make_float4(tf32_round(__uint_as_float(r[j])), tf32_round(__uint_as_float(r[j + 1])),
                                    tf32_round(__uint_as_float(r[j + 2])), tf32_round(__uint_as_float(r[j + 3])));
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == kMmaThread) {
            const uint32_t aXT = smem_u32(s.XT), bM = smem_u32(s.DT);
            for (int ks = 0; ks < C / 8; ++ks)
                umma_tf32(tm + kD4, desc_kmajor(aXT, C, ks), desc_kmajor(bM, C, ks), id64, ks > 0);
            umma_commit(&s.barM[3]);
        }
        // ---- dKt (fp32) and dv (bf16) from product 2: lane = channel c (or v), columns = rows j.
        // Warp (quarter q4, group warp / 4): dKt rows 0..31 | dKt 32..63 | dv 0..31 | dv 32..63.
        // Staged row-major in the stacked operand's tile (product 2 has read it): dKt leaves as
        // one bulk copy, dv as 16-byte pieces of its rows
        ok = ok && mbar_wait(&s.barM[1], par);
        float* const dks = reinterpret_cast<float*>(s.KV);                   // dKt [64 j][128 c]
        uint16_t* const dvs = reinterpret_cast<uint16_t*>(s.KV + kTileCK);   // dv [64 j][128 v]
        if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            const int grp = warp >> 2, c = 32 * q4 + lane, j0 = 32 * (grp & 1);
            uint32_t r[32];
            tmem_ld32_issue(tm + (grp < 2 ? kD2K : kD2V) + ((uint32_t)(32 * q4) << 16) + j0, r);
            tmem_wait_ld(r);
            if (grp < 2) {
#pragma unroll
                for (int j = 0; j < 32; ++j) dks[(j0 + j) * D + c] = __uint_as_float(r[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) dvs[(j0 + j) * D + c] = f2bf(__uint_as_float(r[j]));
            }
        }
        fence_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok);
        if (!ok) break;
        if (tid == 0) {
            bulk_s2g(wy + WyOff::DKT, dks, (uint32_t)kTileCK);
            bulk_commit();
        }
        for (int idx = tid; idx < C * (D / 8); idx += kWyThreads) {
            const int j = idx >> 4, c8 = (idx & 15) * 8;
            if (j < L)
                *reinterpret_cast<uint4*>(dv + ((size_t)(ci.t0 + j) * H + h) * D + c8) =
                    *reinterpret_cast<const uint4*>(dvs + j * D + c8);
        }
        __syncthreads();   // the dv rows are read: the next tile's raw v rows may overwrite them
        // the stacked operand is read: the next tile's K~ and raw v rows stream into its place
        // (K~ once the dKt copy has read its staging)
        if (cn.L > 0) {
            if (tid == 0) { bulk_wait_read_all(); issue_K(nxt); ++nb[2]; }
            stage_v(nxt, cn);
        }
        // ---- dA = -strict_lower(X^T M), dB = diag(beta) dA, dbeta_i += sum_{j<i} dA_ij B_ij
        ok = ok && mbar_wait(&s.barM[3], par);
        if (tid == 0) ok = ok && mbar_wait(&s.barB, par);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        tc_fence_after();
        // dA rows from TMEM (warps 0..7, a row per lane) into the free M tile, its 16-byte
        // chunks swizzled by the row (chunk j/4 ^ (i & 7)), so that both the row-per-lane
        // writes and the row-wise reads below are free of bank conflicts
        float* const dAs = reinterpret_cast<float*>(s.DT);
        auto dA_at = [](int i, int j) { return i * C + ((((j >> 2) ^ (i & 7))) << 2) + (j & 3); };
        if (warp < 8) {
            const int hcol = warp >> 2;
            uint32_t r[32];
            tmem_ld32_issue(tm + kD4 + ((uint32_t)(32 * q4) << 16) + 32 * hcol, r);
            tmem_wait_ld(r);
            if (lrow) {
                const int i = mrow, j0 = 32 * hcol;
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float d[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) d[e] = (j0 + j + e < i) ? -__uint_as_float(r[j + e]) : 0.0f;
                    *reinterpret_cast<float4*>(dAs + dA_at(i, j0 + j)) = make_float4(d[0], d[1], d[2], d[3]);
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        // dB = diag(beta) dA as whole rows (16 lanes x 16 bytes per row), and the row sums of
        // dA_ij B_ij over the 16 lanes of a row in a fixed order
        {
            float* gdB = reinterpret_cast<float*>(wy + WyOff::DB);
            const int jc = tid & 15, j = 4 * jc;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int i = (tid >> 4) + 32 * h2;
                const float4 d = *reinterpret_cast<const float4*>(dAs + dA_at(i, j));
                const float4 bm = *reinterpret_cast<const float4*>(s.Bm + i * C + j);
                const float bi = s.beta[i];
                *reinterpret_cast<float4*>(gdB + i * C + j) = make_float4(bi * d.x, bi * d.y, bi * d.z, bi * d.w);
                float acc = d.x * bm.x + d.y * bm.y + d.z * bm.z + d.w * bm.w;
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (jc == 0) s.db2[i] = acc;
            }
        }
        __syncthreads();
        if (tid < C)
            reinterpret_cast<float*>(wy + WyOff::DBETA)[tid] =
                ((s.dbeta[0][tid] + s.dbeta[1][tid]) + (s.dbeta[2][tid] + s.dbeta[3][tid])) +
                s.db2[tid];
        // B is read: the next tile's B streams in
        if (tid == 0 && cn.L > 0) { issue_B(nxt); ++nb[4]; }
        if (cn.L <= 0) break;
        tile_i = nxt;
        ci = cn;
        braw = braw_next;
        par ^= 1u;
    }
    cp_async_wait_all();
    if (tid == 0) {
        bulk_wait_all();   // the last dKt copy
        if (!ok) raise_status(ws, KDA_ERR_TIMEOUT);
        // bulk copies still in flight (only after an aborted tile), bounded: the last phase
        // issued on each barrier (phases complete in order)
        uint64_t* bars[5] = {&s.barW, &s.barU, &s.barK, &s.barX, &s.barB};
        for (int i = 0; i < 5; ++i)
            if (nb[i] > 0) mbar_wait(bars[i], (uint32_t)((nb[i] - 1) & 1));
    }
    if (tid == kMmaThread) {   // every MMA issued has completed once this phase flips
        umma_commit(&s.barFin);
        mbar_wait(&s.barFin, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

// The instantiation for the plain or the grouped head layout (template kernels are not
// visible outside this file).
BwdWyKernel bwd_wy_kernel(bool grouped) { return grouped ? kda_bwd_wy_kernel<true> : kda_bwd_wy_kernel<false>; }

}  // namespace kda
