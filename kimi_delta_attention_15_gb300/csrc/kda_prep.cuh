// Per-chunk preprocessing shared by the forward and backward chunk kernels,
// so every kernel recomputes bitwise the same values:
//   q^ = q / sqrt(|q|^2 + 1e-6), k^ likewise          (flashinfer contract)
//   beta = sigmoid(beta_raw)
//   alpha_c = exp(lb * sigmoid(exp(A_log) (g_raw_c + dt_bias_c)))   per key channel
// and, per 16-row sub-block I and key channel c, products of alpha:
//   E-_i = prod_{s_I <= j <= i} alpha_j   (decay from the block start, inclusive)
//   E+_i = prod_{i < j <= e_I} alpha_j    (decay to the block end, exclusive)
//   D_I  = prod over the block;  Pb_I = prod_{I' < I} D_I'  (= Gamma at the block start)
//   Sf_I = prod_{I' > I} D_I';  gl = prod_I D_I = exp(G_L)
//   f_IJ = prod_{J < I' < I} D_I' (I > J),  1 / D_I (I = J)
// so that e^{G_i - G_j} = (E-_i f_IJ) (E+_j) for i in block I >= J, j in block J,
// with both factors in [e^{-80}, e^{80}] when lb >= -5. Rows at or past the
// chunk length L are zero with alpha = 1 (no decay) and beta = 0.
#pragma once
#include "kda_internal.cuh"
#include "umma.cuh"

namespace kda {

constexpr int PS = 132;   // padded row stride (floats) of [64][128] smem tiles
constexpr int PC = 68;    // padded row stride of [64][64] smem tiles

struct Factors {
    float F[NSUB][NSUB][D];
    float Pb[NSUB][D];
    float Sf[NSUB][D];
    float Db[NSUB][D];
    float gl[D];
};

// Sum of squares of four consecutive channels, in one fixed fused order.
__device__ __forceinline__ float sq4(float a, float b, float c, float d) {
    return fmaf(d, d, fmaf(c, c, fmaf(b, b, a * a)));
}

// Raw bf16 rows of one chunk held in registers: with NW warps, warp w holds
// rows w + NW b, lane l channels 4l .. 4l+3. The kernels stage a tile's rows in
// shared memory ahead of use and fill these registers from there.
template <int NW>
struct RowRegsT {
    static constexpr int RB = C / NW;
    uint2 q[RB], k[RB], g[RB];
    float br[RB];
    float dt[4];     // dt_bias[h, 4 lane .. 4 lane + 3]
};

// A chunk's rows from raw bf16 copies in shared memory (q, k, g_raw as
// [64][128], beta_raw [64], dt_bias [128] of the head; any may be null; rows at
// or past L read as zero).
template <int NW>
__device__ __forceinline__ void prep_load_staged(RowRegsT<NW>& rr, const uint16_t* qs, const uint16_t* ks,
                                                 const uint16_t* gs, const uint16_t* bs, const float* dtb, int L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = lane * 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) rr.dt[e] = dtb ? dtb[c0 + e] : 0.0f;
#pragma unroll
    for (int b = 0; b < RowRegsT<NW>::RB; ++b) {
        const int r = warp + b * NW;
        rr.q[b] = rr.k[b] = rr.g[b] = make_uint2(0u, 0u);
        rr.br[b] = 0.0f;
        if (r < L) {
            if (qs) rr.q[b] = *reinterpret_cast<const uint2*>(qs + r * D + c0);
            if (ks) rr.k[b] = *reinterpret_cast<const uint2*>(ks + r * D + c0);
            if (gs) rr.g[b] = *reinterpret_cast<const uint2*>(gs + r * D + c0);
            if (bs && lane == 0) rr.br[b] = bf2f(bs[r]);
        }
    }
}

// Turns loaded rows into q^, k^, alpha, beta and 1/sqrt(|x|^2 + eps) in shared
// memory (any output pointer may be null; rows >= L: zeros, alpha = 1, beta = 0).
template <int NW>
__device__ __forceinline__ void prep_compute(const RowRegsT<NW>& rr, float a_h, float lb, int L, float* xq,
                                             float* xk, float* xa, float* beta, float* inq, float* ink) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = lane * 4;
    const float* dtv = rr.dt;
    auto un = [](uint2 w, float* out) {
        out[0] = bf2f((uint16_t)(w.x & 0xffffu)); out[1] = bf2f((uint16_t)(w.x >> 16));
        out[2] = bf2f((uint16_t)(w.y & 0xffffu)); out[3] = bf2f((uint16_t)(w.y >> 16));
    };
    // squared norms of all rows first, then the reductions interleaved across rows.
    // Fixed order: a fused chain over each lane's 4 channels, a butterfly over the 16
    // lanes of each 64-channel half, then the two halves (the pair-term kernel, which
    // splits the channels between two CTAs, forms the same sums bit for bit)
    constexpr int RB = RowRegsT<NW>::RB;
    float sq[RB], sk[RB];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
        float qv[4], kv[4];
        un(rr.q[b], qv); un(rr.k[b], kv);
        sq[b] = sq4(qv[0], qv[1], qv[2], qv[3]);
        sk[b] = sq4(kv[0], kv[1], kv[2], kv[3]);
    }
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        const int o = i < 4 ? 8 >> i : 16;
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            sq[b] += __shfl_xor_sync(0xffffffffu, sq[b], o);
            sk[b] += __shfl_xor_sync(0xffffffffu, sk[b], o);
        }
    }
#pragma unroll
    for (int b = 0; b < RB; ++b) {
        const int r = warp + b * NW;
        float qv[4], kv[4], gr[4], al[4] = {1, 1, 1, 1};
        un(rr.q[b], qv); un(rr.k[b], kv); un(rr.g[b], gr);
        if (xa && r < L) {
#pragma unroll
            for (int e = 0; e < 4; ++e) al[e] = __expf(lb * sigmoidf(a_h * (gr[e] + dtv[e])));
        }
        const float iq = rsqrtf(sq[b] + 1e-6f), ik = rsqrtf(sk[b] + 1e-6f);
        if (xq) *reinterpret_cast<float4*>(xq + r * PS + c0) = make_float4(qv[0] * iq, qv[1] * iq, qv[2] * iq, qv[3] * iq);
        if (xk) *reinterpret_cast<float4*>(xk + r * PS + c0) = make_float4(kv[0] * ik, kv[1] * ik, kv[2] * ik, kv[3] * ik);
        if (xa) *reinterpret_cast<float4*>(xa + r * PS + c0) = make_float4(al[0], al[1], al[2], al[3]);
        if (lane == 0) {
            if (beta) beta[r] = r < L ? sigmoidf(rr.br[b]) : 0.0f;
            if (inq) inq[r] = iq;
            if (ink) ink[r] = ik;
        }
    }
}

// Block products. On entry `ap` holds alpha, `xq`/`xk` hold q^/k^ (either may
// be null). On exit: ap = k^ * E+ (needs xk), xq = q^ * E-, xk = k^ * E-;
// em/ep (nullable) receive E-/E+; fa->Db receives D_I.
__device__ __forceinline__ void block_products(float* ap, float* xq, float* xk, float* em_out, float* ep_out,
                                               Factors* fa) {
    for (int task = threadIdx.x; task < NSUB * D; task += blockDim.x) {
        const int c = task & (D - 1), I = task >> 7;
        float al[SUB], em[SUB], ep[SUB];
#pragma unroll
        for (int i = 0; i < SUB; ++i) al[i] = ap[(I * SUB + i) * PS + c];
        float pre = 1.0f;
#pragma unroll
        for (int i = 0; i < SUB; ++i) { pre *= al[i]; em[i] = pre; }
        float suf = 1.0f;
#pragma unroll
        for (int i = SUB - 1; i >= 0; --i) { ep[i] = suf; suf *= al[i]; }
        fa->Db[I][c] = pre;
#pragma unroll
        for (int i = 0; i < SUB; ++i) {
            const int r = (I * SUB + i) * PS + c;
            if (xk) {
                const float kh = xk[r];
                xk[r] = kh * em[i];
                ap[r] = kh * ep[i];
            }
            if (xq) xq[r] = xq[r] * em[i];
            if (em_out) em_out[r] = em[i];
            if (ep_out) ep_out[r] = ep[i];
        }
    }
}

// Per-channel block factors from fa->Db (threads 0..127). Call after a barrier.
__device__ __forceinline__ void block_factors(Factors* fa) {
    const int c = threadIdx.x;
    if (c >= D) return;
    const float d0 = fa->Db[0][c], d1 = fa->Db[1][c], d2 = fa->Db[2][c], d3 = fa->Db[3][c];
    fa->Pb[0][c] = 1.0f; fa->Pb[1][c] = d0; fa->Pb[2][c] = d0 * d1; fa->Pb[3][c] = d0 * d1 * d2;
    fa->gl[c] = d0 * d1 * d2 * d3;
    fa->Sf[3][c] = 1.0f; fa->Sf[2][c] = d3; fa->Sf[1][c] = d2 * d3; fa->Sf[0][c] = d1 * d2 * d3;
    fa->F[0][0][c] = 1.0f / d0; fa->F[1][1][c] = 1.0f / d1; fa->F[2][2][c] = 1.0f / d2; fa->F[3][3][c] = 1.0f / d3;
    fa->F[1][0][c] = 1.0f; fa->F[2][1][c] = 1.0f; fa->F[3][2][c] = 1.0f;
    fa->F[2][0][c] = d1; fa->F[3][1][c] = d2; fa->F[3][0][c] = d1 * d2;
}

// Decode the t-th lower-triangular block pair (I >= J) of the 4x4 sub-block grid.
__device__ __forceinline__ void tri_pair(int t, int& I, int& J) {
    I = 0;
    while (t > I) { t -= I + 1; ++I; }
    J = t;
}

}  // namespace kda

namespace kda {
// Asynchronous copy of a row-major fp32 [rows][cols] global tile into a padded
// shared tile (row stride `ld` floats); cols a multiple of 4.
__device__ __forceinline__ void tile_to_smem_async(float* dst, int ld, const float* src, int rows, int cols) {
    const int chunks = cols >> 2;
    for (int i = threadIdx.x; i < rows * chunks; i += blockDim.x) {
        const int r = i / chunks, j = i - r * chunks;
        cp_async16(dst + r * ld + 4 * j, src + r * cols + 4 * j);
    }
}
// The same from a [64][128] panel image (umma.cuh layout, R = 64 rows).
__device__ __forceinline__ void panels_to_smem_async(float* dst, int ld, const uint8_t* src) {
    for (int i = threadIdx.x; i < C * 32; i += blockDim.x) {
        const int r = i >> 5, j = i & 31;   // 16-byte chunk j of row r
        cp_async16(dst + r * ld + 4 * j, src + (j >> 3) * C * 128 + r * 128 + ((((j & 7) ^ (r & 7))) << 4));
    }
}
}  // namespace kda
