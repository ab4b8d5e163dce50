// Backward through the UT transform of each chunk: persistent CTAs (one per
// SM) over all (chunk, head) tiles. With W = T (K^*Gamma), U = T V, T = X diag(beta),
// X = (I + A)^{-1}, A = diag(beta) B, and the adjoints dW (state-products
// kernel) and dU = dUt (backward scan):
//   dT    = dW (K^*Gamma)^T + dU V^T
//   dKt   = T^T dW        (adjoint of K^*Gamma)
//   dV    = T^T dU        (final dv)
//   dbeta_j  = sum_i dT_ij X_ij + sum_l dA_jl B_jl
//   dA    = -strict_lower(X^T dT T^T),   dB = diag(beta) dA
// Single tf32 mma.sync products on 16-row tiles: with them every output stays well
// inside its tolerance (measured against the fp64 reference; the pair-term kernel is
// the one that needs split operands); dKt, dB and dbeta go to the workspace.
// The raw k, v, g_raw rows of the CTA's next tile are staged by cp.async during
// the second half of a tile, so the input preparation reads shared memory.
// Warps take row blocks skewed by their index (block (w + w/4) mod 4), so the
// triangular products spread over the four SM sub-partitions evenly.
#include "kda_internal.cuh"
#include "kda_prep.cuh"
#include "mma_sync.cuh"
#include "umma.cuh"

namespace kda {

namespace {
constexpr int VP = D + 8;   // bf16 row pitch of the staged v rows (conflict-free fragment loads)
struct WySmem {
    float kt[C * PS];    // k^, then K^*Gamma
    float dW[C * PS];    // alpha scratch, then dW, then M = dT T^T (stride PC)
    float dU[C * PS];    // dU; after the dKt step the next tile's raw k, g_raw rows
    uint16_t vb[2][C * VP];   // raw v rows (bf16, exact in tf32), by tile parity
    float X[C * PC];
    float B[C * PC];
    float T[C * PC];
    float dT[C * PC];    // dT, then dA
    Factors fa;
    float dtb[D];        // dt_bias of the staged tile's head
    float beta[C];
    float dbeta[C];
    uint16_t braw[C];
};
static_assert(C * PS * 4 >= 2 * C * D * 2, "the staged rows fit in dU");
}  // namespace

size_t bwd_wy_smem_bytes() { return sizeof(WySmem); }

constexpr int kWyWarps = 16;

// kGrouped: k holds H / G heads (grouped value heads); the plain layout is its own
// instantiation so that it carries no head-group arithmetic.
template <bool kGrouped>
__global__ void __launch_bounds__(kWyWarps * 32, 1)
    kda_bwd_wy_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                      const uint16_t* __restrict__ g_raw, const uint16_t* __restrict__ beta_raw,
                      const float* __restrict__ A_log, const float* __restrict__ dt_bias, int H, float lb,
                      uint16_t* __restrict__ dv, uint8_t* __restrict__ ws, Layout lay) {
    extern __shared__ uint8_t smem_raw[];
    WySmem& s = *reinterpret_cast<WySmem*>(smem_raw);
    if (read_status(ws) != 0) return;
    const ChunkInfo* chunks = reinterpret_cast<const ChunkInfo*>(ws + lay.chunks);
    const int ntiles = (int)lay.nc_max * H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    // Persistent over tiles (tile = chunk * H + h). Empty chunk records only
    // follow the last real chunk, so the first empty tile ends the CTA's work.
    const int step = (int)gridDim.x;
    const int G = kGrouped ? (int)lay.G : 1, Hqk = H / G;   // k has Hqk heads
    int tile_i = blockIdx.x;
    ChunkInfo ci = tile_i < ntiles ? chunks[tile_i / H] : ChunkInfo{0, 0, 0, 0};
    if (ci.L <= 0) return;
    uint16_t* const stg = reinterpret_cast<uint16_t*>(s.dU);   // staged k, g_raw rows
    float alog_next = 0.0f;
    uint16_t braw_next = 0;
    // raw rows of tile t_i (record cn) -> staging and vdst; rows past the chunk read as zero
    auto stage_tile = [&](int t_i, const ChunkInfo& cn, uint16_t* vdst) {
        const int hn = t_i % H, hq = hn / G;   // value head, its query/key head
        for (int seg = tid; seg < 3 * C * (D / 8); seg += kWyWarps * 32) {
            const int which = seg >> 10, rem = seg & 1023, r = rem >> 4, c8 = (rem & 15) * 8;
            const uint16_t* src = which == 0 ? k : which == 1 ? g_raw : v;
            const bool valid = r < cn.L;
            // k belongs to query/key head hq (grouped value heads), the rest to value head hn
            const int hs = which == 0 ? hq : hn, Hs = which == 0 ? Hqk : H;
            src += ((size_t)(cn.t0 + (valid ? r : 0)) * Hs + hs) * D + c8;
            uint16_t* dst = which < 2 ? stg + which * C * D + r * D + c8 : vdst + r * VP + c8;
            cp_async16_zfill(dst, src, valid);
        }
        if (tid < D / 4) cp_async16(s.dtb + 4 * tid, dt_bias + (size_t)hn * D + 4 * tid);
        cp_async_commit();
        alog_next = A_log[hn];
        if (tid < C) braw_next = tid < cn.L ? beta_raw[(size_t)(cn.t0 + tid) * H + hn] : (uint16_t)0;
    };
    stage_tile(tile_i, ci, s.vb[0]);
    float alog = alog_next;
    uint16_t braw = braw_next;
    int par = 0;
    while (true) {
    const int nxt = tile_i + step;
    const ChunkInfo cn = nxt < ntiles ? chunks[nxt / H] : ChunkInfo{0, 0, 0, 0};
    const int h = tile_i % H;
    const int L = ci.L;
    const size_t tile = (size_t)tile_i;
    const uint8_t* img = ws + lay.img + tile * ImgOff::BYTES;
    const uint8_t* bg = ws + lay.bg + tile * BgOff::BYTES;
    const uint8_t* gdU = ws + lay.dut + tile * kTileCK;
    uint8_t* wy = ws + lay.wy + tile * WyOff::BYTES;
    const float a_h = __expf(alog);
    const uint16_t* vv = s.vb[par];

    if (tid < C) s.braw[tid] = braw;
    cp_async_wait_all();
    __syncthreads();
    // X, B, then (once the staged rows are read) dU arrive while the rows are prepared
    tile_to_smem_async(s.X, PC, reinterpret_cast<const float*>(img + ImgOff::XM), C, C);
    tile_to_smem_async(s.B, PC, reinterpret_cast<const float*>(img + ImgOff::BM), C, C);
    {
        RowRegsT<kWyWarps> rr;
        prep_load_staged(rr, nullptr, stg, stg + C * D, s.braw, s.dtb, L);
        __syncthreads();
        panels_to_smem_async(s.dU, PS, gdU);
        cp_async_commit();
        prep_compute(rr, a_h, lb, L, nullptr, s.kt, s.dW, s.beta, nullptr, nullptr);
    }
    __syncthreads();
    block_products(s.dW, nullptr, s.kt, nullptr, nullptr, &s.fa);
    __syncthreads();
    block_factors(&s.fa);
    __syncthreads();   // alpha scratch (dW) is free
    tile_to_smem_async(s.dW, PS, reinterpret_cast<const float*>(bg + BgOff::DW), C, D);
    cp_async_commit();
    for (int idx = tid; idx < C * D; idx += blockDim.x) {
        const int r = idx >> 7, c = idx & 127;
        s.kt[r * PS + c] *= s.fa.Pb[r >> 4][c];
    }
    cp_async_wait_all();
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += blockDim.x) {
        const int r = idx >> 6, c = idx & 63;
        s.T[r * PC + c] = s.X[r * PC + c] * s.beta[c];
    }
    __syncthreads();

    // dT = dW Kt^T + dU V^T   (rows 16rb, columns 16ch: 2 n-tiles)
    {
        const int rb = warp & 3, ch = warp >> 2;
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
        for (int ks = 0; ks < D / 8; ++ks) {
            const int k0 = ks * 8 + tig, k1 = k0 + 4;
            const Frag4t wf = ldsm_a(s.dW, PS, rb * SUB, ks * 8);
            const Frag4t uf = ldsm_a(s.dU, PS, rb * SUB, ks * 8);
            Frag2t kb[2];
            ldsm_b2(kb[0], kb[1], s.kt, PS, ch * 16, ks * 8);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int j = ch * 16 + nt * 8 + gid;
                mma1(acc[nt], wf, kb[nt]);
                // v is bf16 data: its fp32 bit pattern is exact in tf32
                mma1(acc[nt], uf, (uint32_t)vv[j * VP + k0] << 16, (uint32_t)vv[j * VP + k1] << 16);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = rb * SUB + gid + (e >> 1) * 8, col = ch * 16 + nt * 8 + tig * 2 + (e & 1);
                s.dT[row * PC + col] = acc[nt][e];
            }
    }
    // dKt = T^T dW, dV = T^T dU   (rows j in 16jb, columns 32ch: 4 n-tiles); T[i][j] = 0 for i < j
    {
        const int jb = (warp + (warp >> 2)) & 3, ch = warp >> 2;
        float ak[4][4], av[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) { ak[nt][e] = 0.0f; av[nt][e] = 0.0f; }
        const int j0 = jb * SUB + gid, j1 = j0 + 8;
        for (int ks = 2 * jb; ks < C / 8; ++ks) {
            const int i0 = ks * 8 + tig, i1 = i0 + 4;
            const Frag4t tf = frag4t(s.T[i0 * PC + j0], s.T[i0 * PC + j1], s.T[i1 * PC + j0], s.T[i1 * PC + j1]);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int c = ch * 32 + nt * 8 + gid;
                mma1(ak[nt], tf, frag2t(s.dW[i0 * PS + c], s.dW[i1 * PS + c]));
                mma1(av[nt], tf, frag2t(s.dU[i0 * PS + c], s.dU[i1 * PS + c]));
            }
        }
        float* gdK = reinterpret_cast<float*>(wy + WyOff::DKT);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = jb * SUB + gid + hh * 8, col = ch * 32 + nt * 8 + tig * 2;
                *reinterpret_cast<float2*>(gdK + row * D + col) = make_float2(ak[nt][hh * 2], ak[nt][hh * 2 + 1]);
                if (row < L) {
                    const uint32_t pk = (uint32_t)f2bf(av[nt][hh * 2]) | ((uint32_t)f2bf(av[nt][hh * 2 + 1]) << 16);
                    *reinterpret_cast<uint32_t*>(dv + ((size_t)(ci.t0 + row) * H + h) * D + col) = pk;
                }
            }
    }
    __syncthreads();
    // k^, v and dU are no longer read: the next tile's rows stream in
    if (cn.L > 0) stage_tile(nxt, cn, s.vb[par ^ 1]);
    // dbeta from T = X diag(beta), sum_{i >= j} dT_ij X_ij: eight threads per column j
    // (rows i = p mod 8), combined by shuffles in a fixed order; M = dT T^T into the dW buffer
    {
        const int j = tid >> 3, p = tid & 7;
        float acc = 0.0f;
#pragma unroll
        for (int i = p; i < C; i += 8)
            if (i >= j) acc += s.dT[i * PC + j] * s.X[i * PC + j];
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (p == 0) s.dbeta[j] = acc;
    }
    float* M = s.dW;
    {
        const int rb = warp & 3, ch = warp >> 2;
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
        for (int ks = 0; ks < C / 8; ++ks) {
            const Frag4t af = ldsm_a(s.dT, PC, rb * SUB, ks * 8);
            Frag2t tb[2];
            ldsm_b2(tb[0], tb[1], s.T, PC, ch * 16, ks * 8);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma1(acc[nt], af, tb[nt]);
        }
        __syncthreads();   // everyone is done reading dW before M overwrites it
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = rb * SUB + gid + (e >> 1) * 8, col = ch * 16 + nt * 8 + tig * 2 + (e & 1);
                M[row * PC + col] = acc[nt][e];
            }
    }
    __syncthreads();
    // dA = -strict_lower(X^T M) into the dT buffer; X[m][i] = 0 for m < i
    {
        const int ib = (warp + (warp >> 2)) & 3, ch = warp >> 2;
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
        const int i0 = ib * SUB + gid, i1 = i0 + 8;
        for (int ks = 2 * ib; ks < C / 8; ++ks) {
            const int m0 = ks * 8 + tig, m1 = m0 + 4;
            const Frag4t xf = frag4t(s.X[m0 * PC + i0], s.X[m0 * PC + i1], s.X[m1 * PC + i0], s.X[m1 * PC + i1]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int j = ch * 16 + nt * 8 + gid;
                mma1(acc[nt], xf, frag2t(M[m0 * PC + j], M[m1 * PC + j]));
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = ib * SUB + gid + (e >> 1) * 8, col = ch * 16 + nt * 8 + tig * 2 + (e & 1);
                s.dT[row * PC + col] = col < row ? -acc[nt][e] : 0.0f;
            }
    }
    __syncthreads();
    float* gdB = reinterpret_cast<float*>(wy + WyOff::DB);
    for (int idx = tid; idx < C * C; idx += blockDim.x) {
        const int r = idx >> 6, c = idx & 63;
        gdB[idx] = s.beta[r] * s.dT[r * PC + c];
    }
    {   // dbeta_i += sum_{j < i} dA_ij B_ij: eight threads per row i, as above
        const int i = tid >> 3, p = tid & 7;
        float acc = 0.0f;
#pragma unroll
        for (int j = p; j < C; j += 8)
            if (j < i) acc += s.dT[i * PC + j] * s.B[i * PC + j];
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (p == 0) reinterpret_cast<float*>(wy + WyOff::DBETA)[i] = s.dbeta[i] + acc;
    }
    if (cn.L <= 0) break;
    tile_i = nxt;
    ci = cn;
    par ^= 1;
    alog = alog_next;
    braw = braw_next;
    }
}

// The instantiation for the plain or the grouped head layout (template kernels are not
// visible outside this file).
BwdWyKernel bwd_wy_kernel(bool grouped) { return grouped ? kda_bwd_wy_kernel<true> : kda_bwd_wy_kernel<false>; }

}  // namespace kda
