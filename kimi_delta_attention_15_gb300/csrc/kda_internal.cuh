// Internal definitions shared by the KDA kernels: chunk geometry, workspace
// layout, device status word, small math helpers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/kda.h"

namespace kda {

constexpr int D = 128;         // K = V = 128
constexpr int C = 64;          // chunk length
constexpr int SUB = 16;        // sub-block length inside a chunk
constexpr int NSUB = C / SUB;  // sub-blocks per chunk

// Per-tile (chunk, head) image sizes in the workspace, bytes.
constexpr size_t kTileCK = (size_t)C * D * 4;     // [64][128] fp32
constexpr size_t kTileCC = (size_t)C * C * 4;     // [64][64]  fp32
constexpr size_t kTileDD = (size_t)D * D * 4;     // [128][128] fp32

// Forward intra-chunk images per tile, written by the intra-chunk kernel.
// "panels" = the 128-byte-swizzled K-major operand layout of umma.cuh
// (values rounded to tf32); R = rows of the image.
//   read by the forward scan:
//     W    [64][128]  panels R=64    W = T (K^ * Gamma)
//     QB   [64][128]  panels R=64    Q^ * Gamma
//     KBT  [128][64]  panels R=128   (K^ * exp(G_L - G))^T
//     AQK  [64][64]   panels R=64    Aqk (decayed q^.k^, j <= i)
//     U    [64][128]  row-major fp32 U = T V (not rounded)
//     GAML [128]      fp32           exp(G_L)
//   read by the backward scan:
//     WT   [128][64]  panels R=128   W^T
//     QBT  [128][64]  panels R=128   scale * (Q^ * Gamma)^T
//     KB   [64][128]  panels R=64    K^ * exp(G_L - G)
//     AQKT [64][64]   panels R=64    scale * Aqk^T
//   read by the backward chunk kernels:
//     XM   [64][64]   row-major fp32 X = (I + A)^{-1}
//     BM   [64][64]   row-major fp32 B_ij = sum_c k^_ic k^_jc e^{G_ic - G_jc} (j < i), A = diag(beta) B
//     KT   [64][128]  panels R=64    K^ * Gamma (the WY backward's operand)
struct ImgOff {
    static constexpr size_t W = 0;
    static constexpr size_t QB = W + kTileCK;
    static constexpr size_t KBT = QB + kTileCK;
    static constexpr size_t AQK = KBT + kTileCK;
    static constexpr size_t FWD_BULK = AQK + kTileCC;   // bytes bulk-loaded by the forward scan
    static constexpr size_t U = FWD_BULK;
    static constexpr size_t GAML = U + kTileCK;
    static constexpr size_t WT = GAML + 1024;
    static constexpr size_t QBT = WT + kTileCK;
    static constexpr size_t KB = QBT + kTileCK;
    static constexpr size_t AQKT = KB + kTileCK;
    static constexpr size_t BWD_BULK = AQKT + kTileCC - WT;  // bytes bulk-loaded by the backward scan
    static constexpr size_t XM = AQKT + kTileCC;
    static constexpr size_t BM = XM + kTileCC;
    static constexpr size_t KT = BM + kTileCC;
    static constexpr size_t BYTES = KT + kTileCK;
};

// Backward state-product outputs per tile (row-major fp32; dW as K-major panels).
struct BgOff {
    static constexpr size_t DQB = 0;                 // dQbar [64][128]
    static constexpr size_t DW = DQB + kTileCK;      // dW    [64][128] panels R=64
    static constexpr size_t DKB = DW + kTileCK;      // dKbar [64][128]
    static constexpr size_t DAQK = DKB + kTileCK;    // dAqk  [64][64] (scale included)
    static constexpr size_t DGAM = DAQK + kTileCC;   // sum_v dS_L * S0 [128]
    static constexpr size_t BYTES = ((DGAM + D * 4) + 1023) & ~size_t(1023);
};

// Backward WY-kernel outputs per tile (row-major fp32).
struct WyOff {
    static constexpr size_t DKT = 0;                 // d(K^ * Gamma) [64][128]
    static constexpr size_t DB = DKT + kTileCK;      // dB = diag(beta) dA [64][64]
    static constexpr size_t DBETA = DB + kTileCC;    // dbeta [64]
    static constexpr size_t BYTES = ((DBETA + C * 4) + 1023) & ~size_t(1023);
};

struct ChunkInfo {
    int32_t t0;   // first token (global, packed index)
    int32_t L;    // rows in this chunk (1..64); 0 = unused slot
    int32_t n;    // sequence
    int32_t c;    // chunk index inside the sequence
};

struct Layout {
    int64_t nc_max;      // chunk slots
    int64_t H;           // value heads
    size_t status, chunks, seq_first, seq_order;
    size_t img, s0, ut, ds, dut, bg, wy, part;
    size_t total;
    int64_t G;           // value heads per query/key head
    // (kept at 14 fields: kernels that take the layout by value spill registers once it grows)
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline int64_t chunk_slots(int64_t B, int64_t T, int64_t N, bool packed) {
    return packed ? (B * T) / C + N + 1 : B * ((T + C - 1) / C);
}

// Chunk classes (chunk index mod kParamGroups) of the parameter reduction, one CTA each.
constexpr int kParamGroups = 8;
__host__ __device__ inline size_t param_scratch_bytes(int64_t H) {
    return (size_t)H * kParamGroups * (D + 4) * 4 + (size_t)H * 4;
}

__host__ __device__ inline Layout make_layout(int64_t B, int64_t T, int64_t H, int64_t N, bool packed,
                                              int64_t G = 1) {
    Layout l;
    l.nc_max = chunk_slots(B, T, N, packed);
    l.H = H;
    l.G = G;
    const int64_t tiles = l.nc_max * H;
    size_t o = 0;
    l.status = o;      o = align_up(o + 256, 1024);
    l.chunks = o;      o = align_up(o + (size_t)l.nc_max * sizeof(ChunkInfo), 1024);
    l.seq_first = o;   o = align_up(o + (size_t)(N + 1) * 4, 1024);
    l.seq_order = o;   o = align_up(o + (size_t)(N + 1) * 4, 1024);
    l.img = o;         o += (size_t)tiles * ImgOff::BYTES;
    l.s0 = o;          o += (size_t)tiles * kTileDD;   // S0^T  [128 k][128 v] panels (tf32)
    l.ut = o;          o += (size_t)tiles * kTileCK;
    l.ds = o;          o += (size_t)tiles * kTileDD;   // dS_L^T [128 k][128 v] panels (tf32)
    l.dut = o;         o += (size_t)tiles * kTileCK;
    l.bg = o;          o += (size_t)tiles * BgOff::BYTES;
    l.wy = o;          o += (size_t)tiles * WyOff::BYTES;
    l.part = o;        o = align_up(o + (size_t)tiles * (D + 4) * 4, 1024);
    // G > 1: every value head's fp32 share of dq and dk, [B T][H][2][128], summed per group
    o = align_up(o + (G > 1 ? (size_t)(B * T) * H * 2 * D * 4 : 0), 1024);
    // the parameter reduction's per-(head, chunk class) sums and per-head counters (last region)
    o = align_up(o + param_scratch_bytes(H), 1024);
    l.total = o;
    return l;
}

// Offset of the parameter reduction's scratch: [H][kParamGroups][D + 4] fp32 sums, then H
// counters of finished (head, chunk class) CTAs.
__host__ __device__ inline size_t param_scratch_offset(const Layout& l) {
    return l.total - align_up(param_scratch_bytes(l.H), 1024);
}

// Kernels with a plain and a grouped-head instantiation, handed out by host accessors
// in the files that define them.
using FwdIntraKernel = void (*)(const uint16_t*, const uint16_t*, const uint16_t*, const uint16_t*,
                                const uint16_t*, const float*, const float*, int, float, float, uint8_t*, Layout);
using BwdWyKernel = void (*)(const uint16_t*, const uint16_t*, const uint16_t*, const uint16_t*, const float*,
                             const float*, int, float, uint16_t*, uint8_t*, Layout);
using BwdPairKernel = void (*)(const uint16_t*, const uint16_t*, const uint16_t*, const uint16_t*, const float*,
                               const float*, int, float, uint16_t*, uint16_t*, uint16_t*, uint16_t*, uint8_t*,
                               Layout);

// Offset of the grouped-head dq, dk shares: the region right after the parameter partials.
__host__ __device__ inline size_t qk_share_offset(const Layout& l) {
    return align_up(l.part + (size_t)(l.nc_max * l.H) * (D + 4) * 4, 1024);
}


// The status region (the first 256 bytes of the workspace): the device status word at
// byte 0; the forward's provenance stamp, a hash of its shape at byte 8 and the
// "forward complete" word at byte 16 (kFwdDone once the forward's last kernel ran
// without error); at byte 24 the count of forward-scan CTAs that have finished.
constexpr size_t kStampHashOff = 8;
constexpr size_t kStampDoneOff = 16;
constexpr size_t kFwdCountOff = 24;
constexpr uint32_t kFwdDone = 0x4b444146u;

// Device status word helpers (first int32 of the workspace).
__device__ __forceinline__ int read_status(const uint8_t* ws) {
    return *reinterpret_cast<const volatile int*>(ws);
}
__device__ __forceinline__ void raise_status(uint8_t* ws, int code) {
    atomicCAS(reinterpret_cast<int*>(ws), 0, code);
}

__device__ __forceinline__ float bf2f(uint16_t x) { return __uint_as_float(((uint32_t)x) << 16); }
__device__ __forceinline__ uint16_t f2bf(float x) {
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&b);
}

// sigmoid via the CUDA exponential and the fast division (denominator >= 1;
// an infinite denominator gives the correct limit 0)
__device__ __forceinline__ float sigmoidf(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// sigmoid(x) * (1 - sigmoid(x)) = u / (1 + u)^2 with u = exp(-|x|): no
// cancellation in 1 - sigmoid(x) when the sigmoid saturates.
__device__ __forceinline__ float dsigmoidf(float x) {
    const float u = __expf(-fabsf(x));
    const float d = 1.0f + u;
    return __fdividef(u, d * d);
}

}  // namespace kda
