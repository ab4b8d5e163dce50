// Forward intra-chunk kernel: persistent CTAs (one per SM) over all
// (chunk, head) tiles, in parallel. For the chunk's L <= 64 tokens it computes
//   q^, k^ (L2 norm, eps 1e-6), beta = sigmoid(beta_raw),
//   alpha = exp(g), g = lb * sigmoid(exp(A_log) (g_raw + dt_bias))   per key channel,
//   the decays between rows from products of alpha inside 16-row sub-blocks,
//   A_ij = beta_i sum_c k^_ic k^_jc e^{G_ic - G_jc} (j < i),
//   Aqk_ij = sum_c q^_ic k^_jc e^{G_ic - G_jc} (j <= i),
//   T = (I + A)^{-1} diag(beta) by blocked forward substitution,
//   W = T (K^ * Gamma), U = T V,
// and stores the images the two state scans consume (kda_internal.cuh).
// The pairwise products and W, U use split-tf32 operands (mma_sync.cuh): the
// gate gradient of the backward needs them to about 1e-6 relative.
//
// The chunk form is the exact "16-sub-chunk + WY" prefill of the
// kda-neuron-kernels log, with a 64-token chunk. Decay factors between rows i
// and j of different sub-blocks are split at the end of j's sub-block, so each
// factor stays in [e^{-80}, e^{80}] for lb >= -5 (sub-blocks of 16 tokens):
//   e^{G_i - G_j} = (e^{G_i - G_{e_J}}) * (e^{G_{e_J} - G_j}),  e_J = last row of block J.
#include "kda_internal.cuh"
#include "mma_sync.cuh"
#include "umma.cuh"
#include "kda_prep.cuh"

namespace kda {

namespace {

constexpr int P = PS;
constexpr int PA = PC;

struct IntraSmem {
    float qe[C * P];      // q^ * E-
    float ke[C * P];      // k^ * E-
    float kp[C * P];      // alpha, then k^ * E+
    float v[C * P];
    float A[C * PA];      // beta-scaled strictly lower A
    float Aqk[C * PA];
    float X[C * PA];      // (I + A)^{-1}
    float T[C * PA];      // X diag(beta)
    Factors fa;
    float beta[C];
};

}  // namespace

constexpr int kIntraWarps = 16;

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
    // The rows of the next tile are loaded into registers while the current one computes.
    // chunk records are read two tiles ahead
    const int step = (int)gridDim.x;
    auto chunk_of = [&](int t) { return t < ntiles ? chunks[t / H] : ChunkInfo{0, 0, 0, 0}; };
    ChunkInfo ci_next = chunk_of(blockIdx.x), ci_next2 = chunk_of(blockIdx.x + step);
    for (int tile_i = blockIdx.x; tile_i < ntiles; tile_i += gridDim.x) {
    const ChunkInfo ci = ci_next;
    const int h = tile_i % H;
    const int nxt = tile_i + step;
    ci_next = ci_next2;
    ci_next2 = chunk_of(nxt + step);
    if (ci.L <= 0) continue;
    const int L = ci.L;
    const float a_h = __expf(A_log[h]);
    const size_t tile = (size_t)tile_i;
    uint8_t* img = ws + lay.img + tile * ImgOff::BYTES;

    prep_rows<kIntraWarps>(q, k, v, g_raw, beta_raw, dt_bias, a_h, lb, ci.t0, L, H, h, s.qe, s.ke, s.v, s.kp,
                           s.beta, nullptr, nullptr);
    __syncthreads();
    block_products(s.kp, s.qe, s.ke, nullptr, nullptr, &s.fa);
    // zero the blocks above the diagonal of A, Aqk, X
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

    // ---- pairwise decayed products, 16x16 blocks (I >= J), tf32 mma.sync
    for (int task = warp; task < 20; task += kIntraWarps) {
        const int m = task / 10;
        int I, J;
        tri_pair(task % 10, I, J);
        const float* base = m == 0 ? s.ke : s.qe;
        const float* f = s.fa.F[I][J];
        float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
        float acc2[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};   // second chain: odd k-steps
        const int r0 = I * SUB + gid, r1 = r0 + 8;
#pragma unroll 2
        for (int ks = 0; ks < D / 8; ks += 2) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int k0 = (ks + u) * 8 + tig, k1 = k0 + 4;
                const float f0 = f[k0], f1 = f[k1];
                const Frag4 af = frag4(base[r0 * P + k0] * f0, base[r1 * P + k0] * f0, base[r0 * P + k1] * f1,
                                       base[r1 * P + k1] * f1);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int j = J * SUB + nt * 8 + gid;
                    mma3(u == 0 ? acc[nt] : acc2[nt], af, frag2(s.kp[j * P + k0], s.kp[j * P + k1]));
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] += acc2[nt][e];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = I * SUB + gid + (e >> 1) * 8;
                const int col = J * SUB + nt * 8 + tig * 2 + (e & 1);
                const float val = acc[nt][e];
                if (m == 0) {
                    const float b = col < row ? val : 0.0f;
                    s.A[row * PA + col] = b * s.beta[row];
                    reinterpret_cast<float*>(img + ImgOff::BM)[row * C + col] = b;
                } else {
                    s.Aqk[row * PA + col] = col <= row ? val : 0.0f;
                }
            }
    }
    __syncthreads();

    // ---- X = (I + A)^{-1}: diagonal 16x16 blocks by forward substitution
    if (warp < NSUB && lane < SUB) {
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
    __syncthreads();
    // off-diagonal blocks, by distance d from the diagonal (the tasks of a level
    // run on separate warps; split-tf32 products keep fp32-level accuracy):
    //   X_IJ = -X_II * sum_{J <= K' < I} A_IK' X_K'J
    for (int d = 1; d < NSUB; ++d) {
        if (warp < NSUB - d) {
            const int J = warp, I = J + d;
            float* Y = s.T + warp * SUB * PA;   // per-warp [16][16] scratch (T is not yet in use)
            float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
            const int r0 = I * SUB + gid, r1 = r0 + 8;
            for (int ks = 2 * J; ks < 2 * I; ++ks) {
                const int m0 = ks * 8 + tig, m1 = m0 + 4;
                const Frag4 af = frag4(s.A[r0 * PA + m0], s.A[r1 * PA + m0], s.A[r0 * PA + m1], s.A[r1 * PA + m1]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int cc = J * SUB + nt * 8 + gid;
                    mma3(acc[nt], af, frag2(s.X[m0 * PA + cc], s.X[m1 * PA + cc]));
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) Y[(gid + (e >> 1) * 8) * PA + nt * 8 + tig * 2 + (e & 1)] = acc[nt][e];
            __syncwarp();
            float xr[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int m0 = ks * 8 + tig, m1 = m0 + 4;
                const Frag4 af = frag4(s.X[r0 * PA + I * SUB + m0], s.X[r1 * PA + I * SUB + m0],
                                       s.X[r0 * PA + I * SUB + m1], s.X[r1 * PA + I * SUB + m1]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int cc = nt * 8 + gid;
                    mma3(xr[nt], af, frag2(Y[m0 * PA + cc], Y[m1 * PA + cc]));
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    s.X[(I * SUB + gid + (e >> 1) * 8) * PA + J * SUB + nt * 8 + tig * 2 + (e & 1)] = -xr[nt][e];
        }
        __syncthreads();
    }
    // T = X diag(beta); X and the zero upper blocks of B to the workspace
    for (int idx = tid; idx < C * C; idx += blockDim.x) {
        const int r = idx >> 6, cc = idx & 63;
        s.T[r * PA + cc] = s.X[r * PA + cc] * s.beta[cc];
    }
    for (int idx = tid; idx < C * C / 4; idx += blockDim.x) {
        const int r = idx >> 4, cc = (idx & 15) * 4;
        *reinterpret_cast<float4*>(img + ImgOff::XM + (r * C + cc) * 4) = *reinterpret_cast<const float4*>(&s.X[r * PA + cc]);
        if ((cc >> 4) > (r >> 4))
            *reinterpret_cast<float4*>(img + ImgOff::BM + (r * C + cc) * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    // ---- W = T (K^ * Gamma), U = T V   (rows 16rb.., columns 32ch..)
    {
        const int rb = warp & 3, ch = warp >> 2;
        float aw[4][4], au[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) { aw[nt][e] = 0.0f; au[nt][e] = 0.0f; }
        const int ra = rb * SUB + gid, rbb = ra + 8;
        for (int ks = 0; ks < 2 * (rb + 1); ++ks) {
            const int j0 = ks * 8 + tig, j1 = j0 + 4;
            const Frag4 tf = frag4(s.T[ra * PA + j0], s.T[rbb * PA + j0], s.T[ra * PA + j1], s.T[rbb * PA + j1]);
            const float* pb = s.fa.Pb[j0 >> 4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int c = ch * 32 + nt * 8 + gid;
                mma3(aw[nt], tf, frag2(s.ke[j0 * P + c] * pb[c], s.ke[j1 * P + c] * pb[c]));
                // v is bf16 data, exact in tf32
                mma2a(au[nt], tf, tf32_bits(s.v[j0 * P + c]), tf32_bits(s.v[j1 * P + c]));
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

    // ---- elementwise images: Q^*Gamma, K^*exp(G_L - G), Aqk, and their transposes
    //      (16-byte stores: a 16-byte chunk of a panel row is 4 consecutive columns)
    for (int idx = tid; idx < C * D / 4; idx += blockDim.x) {
        const int r = idx >> 5, c = (idx & 31) * 4;          // [64][128], 4 columns per thread
        const float* pb = s.fa.Pb[r >> 4];
        const float* sf = s.fa.Sf[r >> 4];
        float4 qb, kb;
        qb.x = tf32_round(s.qe[r * P + c] * pb[c]);         kb.x = tf32_round(s.kp[r * P + c] * sf[c]);
        qb.y = tf32_round(s.qe[r * P + c + 1] * pb[c + 1]); kb.y = tf32_round(s.kp[r * P + c + 1] * sf[c + 1]);
        qb.z = tf32_round(s.qe[r * P + c + 2] * pb[c + 2]); kb.z = tf32_round(s.kp[r * P + c + 2] * sf[c + 2]);
        qb.w = tf32_round(s.qe[r * P + c + 3] * pb[c + 3]); kb.w = tf32_round(s.kp[r * P + c + 3] * sf[c + 3]);
        *reinterpret_cast<float4*>(img + ImgOff::QB + panel_off(r, c, C)) = qb;
        *reinterpret_cast<float4*>(img + ImgOff::KB + panel_off(r, c, C)) = kb;
    }
    for (int idx = tid; idx < C * D / 4; idx += blockDim.x) {
        const int kk = idx >> 4, c = (idx & 15) * 4;         // [128][64], 4 columns (rows of the source) per thread
        float4 qb, kb;
        float* qp = &qb.x;
        float* kp = &kb.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qp[e] = tf32_round(scale * (s.qe[(c + e) * P + kk] * s.fa.Pb[(c + e) >> 4][kk]));
            kp[e] = tf32_round(s.kp[(c + e) * P + kk] * s.fa.Sf[(c + e) >> 4][kk]);
        }
        *reinterpret_cast<float4*>(img + ImgOff::QBT + panel_off(kk, c, D)) = qb;
        *reinterpret_cast<float4*>(img + ImgOff::KBT + panel_off(kk, c, D)) = kb;
    }
    for (int idx = tid; idx < C * C / 4; idx += blockDim.x) {
        const int r = idx >> 4, c = (idx & 15) * 4;
        const float4 a = make_float4(tf32_round(s.Aqk[r * PA + c]), tf32_round(s.Aqk[r * PA + c + 1]),
                                     tf32_round(s.Aqk[r * PA + c + 2]), tf32_round(s.Aqk[r * PA + c + 3]));
        const float4 at = make_float4(tf32_round(scale * s.Aqk[c * PA + r]), tf32_round(scale * s.Aqk[(c + 1) * PA + r]),
                                      tf32_round(scale * s.Aqk[(c + 2) * PA + r]),
                                      tf32_round(scale * s.Aqk[(c + 3) * PA + r]));
        *reinterpret_cast<float4*>(img + ImgOff::AQK + panel_off(r, c, C)) = a;
        *reinterpret_cast<float4*>(img + ImgOff::AQKT + panel_off(r, c, C)) = at;
    }
    if (tid < D) reinterpret_cast<float*>(img + ImgOff::GAML)[tid] = s.fa.gl[tid];
    __syncthreads();   // shared tiles are rewritten by the next tile
    }
}

size_t fwd_intra_smem_bytes() { return sizeof(IntraSmem); }

}  // namespace kda
