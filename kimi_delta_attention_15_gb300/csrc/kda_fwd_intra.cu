// Forward intra-chunk kernel: persistent CTAs (one per SM) over all
// (chunk, head) tiles, in parallel. For the chunk's L <= 64 tokens it computes
//   q^, k^ (L2 norm, eps 1e-6), beta = sigmoid(beta_raw),
//   alpha = exp(g), g = lb * sigmoid(exp(A_log) (g_raw + dt_bias))   per key channel,
//   the decays between rows from products of alpha inside 16-row sub-blocks,
//   A_ij = beta_i sum_c k^_ic k^_jc e^{G_ic - G_jc} (j < i),
//   Aqk_ij = sum_c q^_ic k^_jc e^{G_ic - G_jc} (j <= i),
//   T = (I + A)^{-1} diag(beta) by blocked forward substitution,
//   W = T (K^ * Gamma), U = T V,
// and stores the images the two state scans and the backward chunk kernels consume
// (kda_internal.cuh).
// W and U use about fp32-accurate products (mma_sync.cuh: tf32 high parts plus bf16
// cross terms for W; for U, T's high part in tf32 and its low part in bf16 against the
// exact bf16 v, two k-steps per bf16 product): the final state and the gate
// gradient of the backward need them. The pairwise products of A and Aqk and the
// off-diagonal blocks of the solve use single tf32 products (the measured output
// errors stay well inside their tolerances).
//
// The chunk form is the exact "16-sub-chunk + WY" prefill of the
// kda-neuron-kernels log, with a 64-token chunk. Decay factors between rows i
// and j of different sub-blocks are split at the end of j's sub-block, so each
// factor stays in [e^{-80}, e^{80}] for lb >= -5 (sub-blocks of 16 tokens):
//   e^{G_i - G_j} = (e^{G_i - G_{e_J}}) * (e^{G_{e_J} - G_j}),  e_J = last row of block J.
//
// Schedule of one tile (16 warps). The raw inputs of the CTA's next tile are
// staged by cp.async while the current tile computes W and U, so the input
// preparation reads shared memory instead of waiting on global loads:
//   prep (staged rows) -> block products -> factors
//   pairs: warps 0..9 the ten A blocks, warps 10..15 six Aqk blocks
//   warps 0..3 solve (I + A)^{-1} | warps 4..11 the other four Aqk blocks, by
//     halves (8 columns each) | warps 12..15 the elementwise images
//   T, X and Aqk images; then next tile's rows -> staging; W, U
#include "kda_internal.cuh"
#include "mma_sync.cuh"
#include "umma.cuh"
#include "kda_prep.cuh"

#include <type_traits>

namespace kda {

namespace {

constexpr int P = PS;
constexpr int PA = PC;
constexpr int VP = D + 8;   // bf16 row pitch of the staged v rows (conflict-free fragment loads)

struct IntraSmem {
    float qe[C * P];      // q^ * E-
    float ke[C * P];      // k^ * E-
    float kp[C * P];      // alpha, then k^ * E+
    // A | Aqk | X are contiguous: from the T step of one tile to the input
    // preparation of the next they hold that tile's raw q, k, g_raw rows
    float A[C * PA];      // beta-scaled strictly lower A
    float Aqk[C * PA];
    float X[C * PA];      // (I + A)^{-1}
    float T[C * PA];      // X diag(beta)
    uint16_t vb[2][C * VP];   // raw v rows (bf16, exact in tf32), by tile parity
    Factors fa;
    float dtb[D];         // dt_bias of the staged tile's head
    float beta[C];
    uint16_t braw[C];
};
static_assert(3 * C * PA * 4 >= 3 * C * D * 2, "the staged rows fit in A | Aqk | X");

__device__ __forceinline__ void bar_solve() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

}  // namespace

constexpr int kIntraWarps = 16;

// kGrouped: q, k hold H / G heads (grouped value heads); the plain layout is its own
// instantiation so that it carries no head-group arithmetic.
template <bool kGrouped>
__global__ void __launch_bounds__(kIntraWarps * 32, 1)
    kda_fwd_intra_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                         const uint16_t* __restrict__ v, const uint16_t* __restrict__ g_raw,
                         const uint16_t* __restrict__ beta_raw, const float* __restrict__ A_log,
                         const float* __restrict__ dt_bias, int H, float lb, float scale,
                         uint8_t* __restrict__ ws, Layout lay) {
    extern __shared__ uint8_t smem_raw[];
    IntraSmem& s = *reinterpret_cast<IntraSmem*>(smem_raw);
    if (read_status(ws) != 0) return;
    const ChunkInfo* chunks = reinterpret_cast<const ChunkInfo*>(ws + lay.chunks);
    const int ntiles = (int)lay.nc_max * H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    // Persistent: this CTA takes tiles blockIdx.x, + gridDim.x, ... (tile = chunk * H + h).
    // Empty chunk records only follow the last real chunk, so the first empty
    // tile ends the CTA's work.
    const int step = (int)gridDim.x;
    const int G = kGrouped ? (int)lay.G : 1, Hqk = H / G;   // q, k have Hqk heads
    int tile_i = blockIdx.x;
    ChunkInfo ci = tile_i < ntiles ? chunks[tile_i / H] : ChunkInfo{0, 0, 0, 0};
    if (ci.L <= 0) return;

    uint16_t* const stg = reinterpret_cast<uint16_t*>(s.A);   // staged q, k, g_raw rows
    float alog_next = 0.0f;
    uint16_t braw_next = 0;
    // raw rows of tile t_i (record cn) -> staging and vdst; rows past the chunk read as zero
    auto stage_tile = [&](int t_i, const ChunkInfo& cn, uint16_t* vdst) {
        const int hn = t_i % H, hq = hn / G;   // value head, its query/key head
        for (int seg = tid; seg < 4 * C * (D / 8); seg += kIntraWarps * 32) {
            const int which = seg >> 10, rem = seg & 1023, r = rem >> 4, c8 = (rem & 15) * 8;
            const uint16_t* src = which == 0 ? q : which == 1 ? k : which == 2 ? g_raw : v;
            const bool valid = r < cn.L;
            // q, k belong to query/key head hq (grouped value heads), the rest to value head hn
            const int hs = which < 2 ? hq : hn, Hs = which < 2 ? Hqk : H;
            src += ((size_t)(cn.t0 + (valid ? r : 0)) * Hs + hs) * D + c8;
            uint16_t* dst = which < 3 ? stg + which * C * D + r * D + c8 : vdst + r * VP + c8;
            cp_async16_zfill(dst, src, valid);
        }
        if (tid < D / 4) cp_async16(s.dtb + 4 * tid, dt_bias + (size_t)hn * D + 4 * tid);
        cp_async_commit();
        alog_next = A_log[hn];
        if (tid < C) braw_next = tid < cn.L ? beta_raw[(size_t)(cn.t0 + tid) * H + hn] : (uint16_t)0;
    };

    // NTN n-tiles (8 columns each, from n-tile nt0) of one 16x16 block of A (m = 0) or
    // Aqk (m = 1), single tf32 products
    auto pair_task = [&](auto ntn, auto mm, int t, uint8_t* img, int nt0) {
        constexpr int NTN = decltype(ntn)::value;
        constexpr int m = decltype(mm)::value;
        int I, J;
        tri_pair(t, I, J);
        const float* base = m == 0 ? s.ke : s.qe;
        const float* f = s.fa.F[I][J];
        float acc[NTN][4], acc2[NTN][4];   // acc2: second chain, odd k-steps
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = acc2[nt][e] = 0.0f;
        const int r0 = I * SUB + gid, r1 = r0 + 8;
#pragma unroll 2
        for (int ks = 0; ks < D / 8; ks += 2) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int k0 = (ks + u) * 8 + tig, k1 = k0 + 4;
                const float f0 = f[k0], f1 = f[k1];
                const Frag4t af = frag4t(base[r0 * P + k0] * f0, base[r1 * P + k0] * f0, base[r0 * P + k1] * f1,
                                         base[r1 * P + k1] * f1);
#pragma unroll
                for (int nt = 0; nt < NTN; ++nt) {
                    const int j = J * SUB + (nt0 + nt) * 8 + gid;
                    mma1(u == 0 ? acc[nt] : acc2[nt], af, frag2t(s.kp[j * P + k0], s.kp[j * P + k1]));
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] += acc2[nt][e];
        // element pairs (columns col, col + 1 of one row): 8-byte shared and global stores
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = I * SUB + gid + hh * 8;
                const int col = J * SUB + (nt0 + nt) * 8 + tig * 2;
                const float v0 = acc[nt][2 * hh], v1 = acc[nt][2 * hh + 1];
                if constexpr (m == 0) {
                    const float b0 = col < row ? v0 : 0.0f, b1 = col + 1 < row ? v1 : 0.0f;
                    const float br = s.beta[row];
                    *reinterpret_cast<float2*>(&s.A[row * PA + col]) = make_float2(b0 * br, b1 * br);
                    *reinterpret_cast<float2*>(img + ImgOff::BM + (row * C + col) * 4) = make_float2(b0, b1);
                } else {
                    *reinterpret_cast<float2*>(&s.Aqk[row * PA + col]) =
                        make_float2(col <= row ? v0 : 0.0f, col + 1 <= row ? v1 : 0.0f);
                }
            }
    };

    stage_tile(tile_i, ci, s.vb[0]);
    float alog = alog_next;
    uint16_t braw = braw_next;
    int par = 0;
    while (true) {
        const int nxt = tile_i + step;
        const ChunkInfo cn = nxt < ntiles ? chunks[nxt / H] : ChunkInfo{0, 0, 0, 0};
        const int L = ci.L;
        const float a_h = __expf(alog);
        uint8_t* img = ws + lay.img + (size_t)tile_i * ImgOff::BYTES;
        if (tid < C) s.braw[tid] = braw;
        cp_async_wait_all();
        __syncthreads();
        {
            RowRegsT<kIntraWarps> rr;
            prep_load_staged(rr, stg, stg + C * D, stg + 2 * C * D, s.braw, s.dtb, L);
            prep_compute(rr, a_h, lb, L, s.qe, s.ke, s.kp, s.beta, nullptr, nullptr);
        }
        __syncthreads();
        block_products(s.kp, s.qe, s.ke, nullptr, nullptr, &s.fa);
        // zero the blocks above the diagonal of A, Aqk, X (the staged rows are consumed)
        for (int idx = tid; idx < C * C; idx += blockDim.x) {
            const int r = idx >> 6, cc = idx & 63;
            if ((cc >> 4) > (r >> 4)) {
                s.A[r * PA + cc] = 0.0f;
                s.Aqk[r * PA + cc] = 0.0f;
                s.X[r * PA + cc] = 0.0f;
            }
        }
        __syncthreads();
        block_factors(&s.fa);
        __syncthreads();

        // ---- pairwise decayed products: all of A first (the solve needs it)
        using Two = std::integral_constant<int, 2>;
        using One = std::integral_constant<int, 1>;
        using BlockA = std::integral_constant<int, 0>;
        using BlockAqk = std::integral_constant<int, 1>;
        if (warp < 10) pair_task(Two{}, BlockA{}, warp, img, 0);
        else pair_task(Two{}, BlockAqk{}, warp - 10, img, 0);
        __syncthreads();

        if (warp < NSUB) {
            // ---- X = (I + A)^{-1}: diagonal 16x16 blocks by forward substitution
            if (lane < SUB) {
                const int I = warp, col = lane;
                float x[SUB];
#pragma unroll
                for (int i = 0; i < SUB; ++i) {
                    float acc = (i == col) ? 1.0f : 0.0f;
#pragma unroll
                    for (int m2 = 0; m2 < i; ++m2) acc -= s.A[(I * SUB + i) * PA + I * SUB + m2] * x[m2];
                    x[i] = acc;
                    s.X[(I * SUB + i) * PA + I * SUB + col] = acc;
                }
            }
            bar_solve();
            // off-diagonal blocks, by distance d from the diagonal:
            //   X_IJ = -X_II * sum_{J <= K' < I} A_IK' X_K'J
            for (int d = 1; d < NSUB; ++d) {
                if (warp < NSUB - d) {
                    const int J = warp, I = J + d;
                    float* Y = s.T + warp * SUB * PA;   // per-warp [16][16] scratch (T is not yet in use)
                    float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
                    const int r0 = I * SUB + gid, r1 = r0 + 8;
                    for (int ks = 2 * J; ks < 2 * I; ++ks) {
                        const int m0 = ks * 8 + tig, m1 = m0 + 4;
                        const Frag4t af =
                            frag4t(s.A[r0 * PA + m0], s.A[r1 * PA + m0], s.A[r0 * PA + m1], s.A[r1 * PA + m1]);
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const int cc = J * SUB + nt * 8 + gid;
                            mma1(acc[nt], af, frag2t(s.X[m0 * PA + cc], s.X[m1 * PA + cc]));
                        }
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            Y[(gid + (e >> 1) * 8) * PA + nt * 8 + tig * 2 + (e & 1)] = acc[nt][e];
                    __syncwarp();
                    float xr[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const int m0 = ks * 8 + tig, m1 = m0 + 4;
                        const Frag4t af = frag4t(s.X[r0 * PA + I * SUB + m0], s.X[r1 * PA + I * SUB + m0],
                                                 s.X[r0 * PA + I * SUB + m1], s.X[r1 * PA + I * SUB + m1]);
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const int cc = nt * 8 + gid;
                            mma1(xr[nt], af, frag2t(Y[m0 * PA + cc], Y[m1 * PA + cc]));
                        }
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            s.X[(I * SUB + gid + (e >> 1) * 8) * PA + J * SUB + nt * 8 + tig * 2 + (e & 1)] =
                                -xr[nt][e];
                }
                bar_solve();
            }
        } else if (warp < 12) {
            pair_task(std::integral_constant<int, 1>{}, std::integral_constant<int, 1>{}, 6 + ((warp - NSUB) >> 1),
                      img, (warp - NSUB) & 1);
        } else {
            // ---- elementwise images: Q^*Gamma, K^*exp(G_L - G), K^*Gamma and the transposes of
            // the first two, by 4x4 blocks (rows 4rb.., columns 4cb..): each thread stores a
            // block's rows and, from the same registers, its columns. A warp takes 4 x 8 blocks
            // (lane: rb += lane / 8, cb += lane % 8): row stores of 128 contiguous bytes and
            // column stores of 64, loads of eight consecutive 16-byte chunks of one row
            const int et = tid - 384, ew = warp - 12;
            for (int g = ew; g < (C / 16) * (D / 32); g += 4) {
                const int rb = 4 * (g >> 2) + (lane >> 3), cb = 8 * (g & 3) + (lane & 7);
                const int r0 = 4 * rb, c0 = 4 * cb;
                const float4 pb = *reinterpret_cast<const float4*>(&s.fa.Pb[r0 >> 4][c0]);
                const float4 sf = *reinterpret_cast<const float4*>(&s.fa.Sf[r0 >> 4][c0]);
                float qb[4][4], kb[4][4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = r0 + e;
                    const float4 qh = *reinterpret_cast<const float4*>(&s.qe[r * P + c0]);
                    const float4 kp = *reinterpret_cast<const float4*>(&s.kp[r * P + c0]);
                    const float4 kh = *reinterpret_cast<const float4*>(&s.ke[r * P + c0]);
                    const float qv[4] = {qh.x * pb.x, qh.y * pb.y, qh.z * pb.z, qh.w * pb.w};
                    const float kv[4] = {kp.x * sf.x, kp.y * sf.y, kp.z * sf.z, kp.w * sf.w};
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        qb[e][f] = tf32_round(scale * qv[f]);   // the transposed image carries the scale
                        kb[e][f] = tf32_round(kv[f]);
                    }
                    *reinterpret_cast<float4*>(img + ImgOff::QB + panel_off(r, c0, C)) =
                        make_float4(tf32_round(qv[0]), tf32_round(qv[1]), tf32_round(qv[2]), tf32_round(qv[3]));
                    *reinterpret_cast<float4*>(img + ImgOff::KB + panel_off(r, c0, C)) =
                        make_float4(kb[e][0], kb[e][1], kb[e][2], kb[e][3]);
                    *reinterpret_cast<float4*>(img + ImgOff::KT + panel_off(r, c0, C)) =
                        make_float4(tf32_round(kh.x * pb.x), tf32_round(kh.y * pb.y), tf32_round(kh.z * pb.z),
                                    tf32_round(kh.w * pb.w));
                }
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    *reinterpret_cast<float4*>(img + ImgOff::QBT + panel_off(c0 + f, r0, D)) =
                        make_float4(qb[0][f], qb[1][f], qb[2][f], qb[3][f]);
                    *reinterpret_cast<float4*>(img + ImgOff::KBT + panel_off(c0 + f, r0, D)) =
                        make_float4(kb[0][f], kb[1][f], kb[2][f], kb[3][f]);
                }
            }
            if (et < D) reinterpret_cast<float*>(img + ImgOff::GAML)[et] = s.fa.gl[et];
        }
        __syncthreads();

        // T = X diag(beta); X, the zero upper blocks of B and the Aqk images to the workspace
        for (int idx = tid; idx < C * C; idx += blockDim.x) {
            const int r = idx >> 6, cc = idx & 63;
            s.T[r * PA + cc] = s.X[r * PA + cc] * s.beta[cc];
        }
        if (warp < 8) {
            // Aqk and (scale Aqk)^T by 4x4 blocks (rows i0.., columns j0..), both from the same
            // registers: row stores of 128 contiguous bytes, column stores of 64
            const int j0 = 4 * ((warp & 1) * 8 + (lane & 7)), i0 = 4 * ((warp >> 1) * 4 + (lane >> 3));
            float av[4][4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 a = *reinterpret_cast<const float4*>(&s.Aqk[(i0 + e) * PA + j0]);
                av[e][0] = a.x; av[e][1] = a.y; av[e][2] = a.z; av[e][3] = a.w;
                *reinterpret_cast<float4*>(img + ImgOff::AQK + panel_off(i0 + e, j0, C)) =
                    make_float4(tf32_round(a.x), tf32_round(a.y), tf32_round(a.z), tf32_round(a.w));
            }
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const float4 at = make_float4(tf32_round(scale * av[0][e2]), tf32_round(scale * av[1][e2]),
                                              tf32_round(scale * av[2][e2]), tf32_round(scale * av[3][e2]));
                *reinterpret_cast<float4*>(img + ImgOff::AQKT + panel_off(j0 + e2, i0, C)) = at;
            }
        } else {
            // X and the zero upper blocks of B (warps 8..15)
            for (int idx = tid - 256; idx < C * C / 4; idx += 256) {
                const int r = idx >> 4, cc = (idx & 15) * 4;
                *reinterpret_cast<float4*>(img + ImgOff::XM + (r * C + cc) * 4) =
                    *reinterpret_cast<const float4*>(&s.X[r * PA + cc]);
                if ((cc >> 4) > (r >> 4))
                    *reinterpret_cast<float4*>(img + ImgOff::BM + (r * C + cc) * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        __syncthreads();

        // the next tile's rows stream in while W and U are formed
        if (cn.L > 0) stage_tile(nxt, cn, s.vb[par ^ 1]);

        // ---- W = T (K^ * Gamma), U = T V   (rows 16rb.., columns 32ch..)
        {
            const uint16_t* vv = s.vb[par];
            // row block skewed by the warp index: the triangular work spreads over
            // the four SM sub-partitions (warp % 4) evenly
            const int rb = (warp + (warp >> 2)) & 3, ch = warp >> 2;
            float aw[4][4], au[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) { aw[nt][e] = 0.0f; au[nt][e] = 0.0f; }
            const int ra = rb * SUB + gid, rbb = ra + 8;
            // k-steps in pairs (the triangle spans an even number): U's low-part products of
            // both steps run as one bf16 m16n8k16 product (v is exact in bf16)
            for (int kq = 0; kq < rb + 1; ++kq) {
                Frag4x tf[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int j0 = (2 * kq + u) * 8 + tig, j1 = j0 + 4;
                    tf[u] = frag4x(s.T[ra * PA + j0], s.T[rbb * PA + j0], s.T[ra * PA + j1], s.T[rbb * PA + j1]);
                }
                const uint32_t alo[4] = {tf[0].bf[2], tf[0].bf[3], tf[1].bf[2], tf[1].bf[3]};
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int c = ch * 32 + nt * 8 + gid;
                    uint32_t vb2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int j0 = (2 * kq + u) * 8 + tig, j1 = j0 + 4;
                        const float* pb = s.fa.Pb[j0 >> 4];
                        mma2x(aw[nt], tf[u], frag2x(s.ke[j0 * P + c] * pb[c], s.ke[j1 * P + c] * pb[c]));
                        const uint32_t v0 = vv[j0 * VP + c], v1 = vv[j1 * VP + c];
                        // v is bf16 data: its fp32 bit pattern is exact in tf32
                        mma_tf32_16x8x8(au[nt], tf[u].hi[0], tf[u].hi[1], tf[u].hi[2], tf[u].hi[3], v0 << 16, v1 << 16);
                        vb2[u] = v0 | (v1 << 16);
                    }
                    mma_bf16_16x8x16(au[nt], alo, vb2);
                }
            }
            float* gU = reinterpret_cast<float*>(img + ImgOff::U);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int row = rb * SUB + gid + hh * 8;
                    const int col = ch * 32 + nt * 8 + tig * 2;
                    const float w0 = tf32_round(aw[nt][hh * 2]), w1 = tf32_round(aw[nt][hh * 2 + 1]);
                    *reinterpret_cast<float2*>(img + ImgOff::W + panel_off(row, col, C)) = make_float2(w0, w1);
                    *reinterpret_cast<float*>(img + ImgOff::WT + panel_off(col, row, D)) = w0;
                    *reinterpret_cast<float*>(img + ImgOff::WT + panel_off(col + 1, row, D)) = w1;
                    *reinterpret_cast<float2*>(gU + row * D + col) = make_float2(au[nt][hh * 2], au[nt][hh * 2 + 1]);
                }
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
FwdIntraKernel fwd_intra_kernel(bool grouped) {
    return grouped ? kda_fwd_intra_kernel<true> : kda_fwd_intra_kernel<false>;
}

size_t fwd_intra_smem_bytes() { return sizeof(IntraSmem); }

}  // namespace kda
