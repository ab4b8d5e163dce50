// One decode step of the gated delta rule for a batch of requests, the recurrence
// of the chunked kernels taken one token at a time. Per (request n, head h), with
// the value-first state S (V x K = 128 x 128 fp32) updated in place:
//   q^ = q / sqrt(|q|^2 + 1e-6), k^ likewise,  beta = sigmoid(beta_raw)
//   alpha_c = exp(lb * sigmoid(exp(A_log[h]) (g_raw_c + dt_bias[h, c])))   per key channel
//   S' = S diag(alpha),  r = v - S' k^,  S = S' + beta r k^T,  o = scale S q^
// Each unit reads and writes its 64 KB state once and does about 1 flop per byte, so
// the step is bound by HBM: the matrix-vector products run on the CUDA cores in fp32.
// One CTA per unit: warp w owns state rows 16w .. 16w+15, lane l key channels
// 4l .. 4l+3 of every one of them (a warp moves whole 512-byte rows); the per-channel
// quantities (alpha, k^, q^) are computed by every warp for its own lanes.
#include <cstdio>
#include "kda_internal.cuh"

namespace kda {
void set_last_error_text(const char* msg);

namespace {
constexpr int kDecRows = 16;   // state rows per warp (8 warps x 16 = 128)

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
}  // namespace

__global__ void __launch_bounds__(256)
    kda_decode_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                      const uint16_t* __restrict__ v, const uint16_t* __restrict__ g_raw,
                      const uint16_t* __restrict__ beta_raw, const float* __restrict__ A_log,
                      const float* __restrict__ dt_bias, float* __restrict__ state, uint16_t* __restrict__ o,
                      int H, int G, float scale, float lb) {
    const int64_t unit = blockIdx.x;   // n * H + h
    const int h = (int)(unit % H);
    // q, k of query/key head h / G (grouped value heads; G = 1: the plain layout)
    const size_t qk = ((size_t)(unit / H) * (H / G) + h / G) * D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = 4 * lane;
    float* S = state + unit * D * D;

    // the state rows of this warp: issued first, they are the bulk of the traffic
    float4 s[kDecRows];
#pragma unroll
    for (int i = 0; i < kDecRows; ++i)
        s[i] = *reinterpret_cast<const float4*>(S + (size_t)(warp * kDecRows + i) * D + c0);

    const size_t tok = (size_t)unit * D;
    const uint2 qw = *reinterpret_cast<const uint2*>(q + qk + c0);
    const uint2 kw = *reinterpret_cast<const uint2*>(k + qk + c0);
    const uint2 gw = *reinterpret_cast<const uint2*>(g_raw + tok + c0);
    const float4 dtb = *reinterpret_cast<const float4*>(dt_bias + (size_t)h * D + c0);
    const float a_h = __expf(A_log[h]);
    const float beta = sigmoidf(bf2f(beta_raw[unit]));
    float vrow[kDecRows];
#pragma unroll
    for (int i = 0; i < kDecRows; ++i) vrow[i] = bf2f(v[tok + warp * kDecRows + i]);

    auto un = [](uint2 w, float* x) {
        x[0] = bf2f((uint16_t)(w.x & 0xffffu)); x[1] = bf2f((uint16_t)(w.x >> 16));
        x[2] = bf2f((uint16_t)(w.y & 0xffffu)); x[3] = bf2f((uint16_t)(w.y >> 16));
    };
    float qv[4], kv[4], gv[4];
    un(qw, qv); un(kw, kv); un(gw, gv);
    const float dt[4] = {dtb.x, dtb.y, dtb.z, dtb.w};
    float sq = 0.0f, sk = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) { sq += qv[e] * qv[e]; sk += kv[e] * kv[e]; }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float iq = rsqrtf(sq + 1e-6f), ik = rsqrtf(sk + 1e-6f);
    float qh[4], kh[4], al[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        qh[e] = qv[e] * iq;
        kh[e] = kv[e] * ik;
        al[e] = __expf(lb * sigmoidf(a_h * (gv[e] + dt[e])));
    }

    // S' = S diag(alpha) and (S' k^)_v for all rows, the reductions interleaved
    float part[kDecRows];
#pragma unroll
    for (int i = 0; i < kDecRows; ++i) {
        s[i].x *= al[0]; s[i].y *= al[1]; s[i].z *= al[2]; s[i].w *= al[3];
        part[i] = s[i].x * kh[0] + s[i].y * kh[1] + s[i].z * kh[2] + s[i].w * kh[3];
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1)
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) part[i] += __shfl_xor_sync(0xffffffffu, part[i], o2);
    // rank-one write, then (S q^)_v
#pragma unroll
    for (int i = 0; i < kDecRows; ++i) {
        const float br = beta * (vrow[i] - part[i]);
        s[i].x += br * kh[0]; s[i].y += br * kh[1]; s[i].z += br * kh[2]; s[i].w += br * kh[3];
        *reinterpret_cast<float4*>(S + (size_t)(warp * kDecRows + i) * D + c0) = s[i];
        part[i] = s[i].x * qh[0] + s[i].y * qh[1] + s[i].z * qh[2] + s[i].w * qh[3];
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1)
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) part[i] += __shfl_xor_sync(0xffffffffu, part[i], o2);
    if (lane < kDecRows) {
        float ov = part[0];
#pragma unroll
        for (int i = 1; i < kDecRows; ++i) ov = lane == i ? part[i] : ov;
        o[tok + warp * kDecRows + lane] = f2bf(scale * ov);
    }
}

}  // namespace kda

extern "C" kda_status kda_decode(long long n_req, long long H, long long groups, float scale, float lower_bound,
                                 const kda_bf16* q, const kda_bf16* k, const kda_bf16* v, const kda_bf16* g_raw,
                                 const kda_bf16* beta_raw, const float* A_log, const float* dt_bias, float* state,
                                 kda_bf16* o, void* stream) {
    if (n_req < 0 || H <= 0 || H > (1 << 20) || n_req * H > (1LL << 31) - 1) return KDA_ERR_SHAPE;
    if (groups < 0 || (groups > 1 && H % groups != 0)) return KDA_ERR_SHAPE;
    const int G = groups > 1 ? (int)groups : 1;
    if (!(scale > 0.0f) || !(scale < 1e30f)) return KDA_ERR_UNSUPPORTED;
    if (!(lower_bound >= -5.0f && lower_bound < 0.0f)) return KDA_ERR_UNSUPPORTED;
    if (n_req == 0) return KDA_OK;
    if (!q || !k || !v || !g_raw || !beta_raw || !A_log || !dt_bias || !state || !o) return KDA_ERR_NULL;
    const void* ptrs[] = {q, k, v, g_raw, beta_raw, A_log, dt_bias, state, o};
    for (const void* p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) & 15u) return KDA_ERR_ALIGN;
    kda::kda_decode_kernel<<<(unsigned)(n_req * H), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint16_t*>(k),
        reinterpret_cast<const uint16_t*>(v), reinterpret_cast<const uint16_t*>(g_raw),
        reinterpret_cast<const uint16_t*>(beta_raw), A_log, dt_bias, state, reinterpret_cast<uint16_t*>(o),
        (int)H, G, scale, lower_bound);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[160];
        snprintf(msg, sizeof(msg), "kda_decode launch: %s (%d)", cudaGetErrorString(e), (int)e);
        kda::set_last_error_text(msg);
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}
