// C ABI entry points (include/kda.h): argument validation, workspace layout,
// the chunk table built on the device from cu_seqlens, and kernel launches.
#include <cmath>
#include <cstdio>
#include <cstring>
#include "kda_internal.cuh"

namespace kda {

size_t fwd_intra_smem_bytes();
size_t fwd_scan_smem_bytes();
size_t bwd_scan_smem_bytes();
size_t bwd_state_smem_bytes();
size_t bwd_wy_smem_bytes();
size_t bwd_pair_smem_bytes();

FwdIntraKernel fwd_intra_kernel(bool grouped);
__global__ void kda_fwd_scan_kernel(const float*, uint16_t*, float*, int, float, uint8_t*, Layout);
__global__ void kda_bwd_scan_kernel(const uint16_t*, const float*, float*, int, uint8_t*, Layout, uint64_t);
__global__ void kda_bwd_state_kernel(const uint16_t*, int, float, uint8_t*, Layout);
BwdWyKernel bwd_wy_kernel(bool grouped);
BwdPairKernel bwd_pair_kernel(bool grouped);
__global__ void kda_param_reduce_kernel(int, float*, float*, uint8_t*, Layout);
__global__ void kda_qk_group_reduce_kernel(uint16_t*, uint16_t*, uint8_t*, int64_t, Layout);

// Chunk table from the offsets: validates cu_seqlens (cu[0] = 0, non-decreasing,
// cu[N] = T_total), lists the chunks of every sequence in order (a chunk never
// crosses a sequence boundary), the first chunk of each sequence, and the
// sequences ordered by decreasing chunk count (longest first, for the scans).
// One CTA; N is small next to the token count.
constexpr int kOrderKeys = 4096;   // distinct chunk counts the scan order tells apart

// It also starts the forward's bookkeeping: clears the status word, stamps the shape hash
// and marks the forward as not complete yet (the forward scan's last CTA completes it).
__global__ void __launch_bounds__(1024)
    kda_chunk_table_kernel(const int64_t* __restrict__ cu, int64_t N, int64_t T_total, int64_t T_fixed,
                           uint8_t* __restrict__ ws, Layout lay, uint64_t shape_hash, int full_workspace) {
    __shared__ int carry;
    __shared__ int bad;
    __shared__ int scan[1024];
    ChunkInfo* chunks = reinterpret_cast<ChunkInfo*>(ws + lay.chunks);
    int* first = reinterpret_cast<int*>(ws + lay.seq_first);
    int* order = reinterpret_cast<int*>(ws + lay.seq_order);
    const int tid = threadIdx.x;
    auto cu_at = [&](int64_t i) -> int64_t { return cu ? cu[i] : i * T_fixed; };
    if (tid == 0) {
        *reinterpret_cast<int*>(ws) = 0;
        *reinterpret_cast<uint64_t*>(ws + kStampHashOff) = shape_hash;
        *reinterpret_cast<uint32_t*>(ws + kStampDoneOff) = 0u;
        *reinterpret_cast<uint32_t*>(ws + kFwdCountOff) = 0u;
        carry = 0;
        bad = (cu_at(0) != 0 || cu_at(N) != T_total) ? 1 : 0;
    }
    // the parameter reduction's counters (the backward's region: full workspaces only)
    if (full_workspace) {
        int* cnt = reinterpret_cast<int*>(ws + param_scratch_offset(lay) + (size_t)lay.H * kParamGroups * (D + 4) * 4);
        for (int64_t i = tid; i < lay.H; i += blockDim.x) cnt[i] = 0;
    }
    __syncthreads();
    for (int64_t b = 0; b < N; b += blockDim.x) {
        const int64_t n = b + tid;
        int nch = 0;
        if (n < N) {
            const int64_t L = cu_at(n + 1) - cu_at(n);
            if (L < 0) atomicOr(&bad, 1);
            nch = L > 0 ? (int)((L + C - 1) / C) : 0;
        }
        scan[tid] = nch;
        __syncthreads();
        for (int off = 1; off < (int)blockDim.x; off <<= 1) {
            const int x = tid >= off ? scan[tid - off] : 0;
            __syncthreads();
            scan[tid] += x;
            __syncthreads();
        }
        const int excl = carry + scan[tid] - nch;
        if (n < N) first[n] = excl;
        __syncthreads();
        if (tid == blockDim.x - 1) carry += scan[tid];
        __syncthreads();
    }
    const int total = carry;
    if (tid == 0) first[N] = total;
    __syncthreads();
    if (bad || total > lay.nc_max) {
        for (int64_t i = tid; i < lay.nc_max; i += blockDim.x) chunks[i] = ChunkInfo{0, 0, 0, 0};
        for (int64_t n = tid; n <= N; n += blockDim.x) first[n] = 0;
        for (int64_t n = tid; n < N; n += blockDim.x) order[n] = (int)n;
        if (tid == 0) raise_status(ws, KDA_ERR_OFFSETS);
        return;
    }
    for (int64_t n = tid; n < N; n += blockDim.x) {
        const int64_t t0 = cu_at(n), L = cu_at(n + 1) - t0;
        const int f = first[n];
        for (int64_t c = 0; c * C < L; ++c) {
            const int64_t rem = L - c * C;
            chunks[f + c] = ChunkInfo{(int32_t)(t0 + c * C), (int32_t)(rem < C ? rem : C), (int32_t)n, (int32_t)c};
        }
    }
    for (int64_t i = total + tid; i < lay.nc_max; i += blockDim.x) chunks[i] = ChunkInfo{0, 0, 0, 0};
    // Scan order, longest sequence first: a counting sort on the chunk count (capped at
    // kOrderKeys - 1), linear in N. Sequences with the same key take any order among
    // themselves: the order only schedules the scans' CTAs, every (sequence, head)
    // result is computed alone, so the outputs do not depend on it.
    __shared__ int slot[kOrderKeys];
    for (int k = tid; k < kOrderKeys; k += blockDim.x) slot[k] = 0;
    __syncthreads();
    auto key_of = [&](int64_t n) { return min(first[n + 1] - first[n], kOrderKeys - 1); };
    for (int64_t n = tid; n < N; n += blockDim.x) atomicAdd(&slot[key_of(n)], 1);
    __syncthreads();
    // slot[k] <- sequences with a larger key (exclusive prefix over descending keys):
    // thread t sums keys 4t .. 4t+3 from the top, then a block scan over the threads
    constexpr int kPer = kOrderKeys / 1024;
    static_assert(kOrderKeys % 1024 == 0, "keys per thread");
    int part[kPer], sum = 0;
    for (int j = 0; j < kPer; ++j) {
        part[j] = slot[kOrderKeys - 1 - (kPer * tid + j)];
        sum += part[j];
    }
    scan[tid] = sum;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int x = tid >= off ? scan[tid - off] : 0;
        __syncthreads();
        scan[tid] += x;
        __syncthreads();
    }
    int run = scan[tid] - sum;
    for (int j = 0; j < kPer; ++j) {
        slot[kOrderKeys - 1 - (kPer * tid + j)] = run;
        run += part[j];
    }
    __syncthreads();
    for (int64_t n = tid; n < N; n += blockDim.x) order[atomicAdd(&slot[key_of(n)], 1)] = (int)n;
}

// Lets the other translation units of the library set the text kda_last_error returns.
void set_last_error_text(const char* msg);

}  // namespace kda

using namespace kda;

namespace {

// Last CUDA error seen by an entry point of this thread (kda_last_error).
thread_local char g_last_error[256] = "";
kda_status cuda_status(cudaError_t e, const char* where) {
    if (e == cudaSuccess) return KDA_OK;
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
    return KDA_ERR_CUDA;
}

// Optional per-kernel timing events (kda_set_profile_events).
const cudaEvent_t* g_prof = nullptr;
int g_prof_n = 0;
inline void prof(int slot, cudaStream_t s) {
    if (g_prof && slot < g_prof_n) cudaEventRecord(g_prof[slot], s);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status check_shape(const kda_shape* sh, bool packed) {
    if (!sh) return KDA_ERR_NULL;
    if (sh->K != 128 || sh->V != 128) return KDA_ERR_UNSUPPORTED;
    if (!(sh->lower_bound >= -5.0f && sh->lower_bound < 0.0f)) return KDA_ERR_UNSUPPORTED;
    if (!(std::isfinite(sh->scale) && sh->scale > 0.0f)) return KDA_ERR_UNSUPPORTED;
    if (sh->B < 1 || sh->T < 0 || sh->H < 1 || sh->H > 65535 || sh->N < 0) return KDA_ERR_SHAPE;
    if (packed) {
        if (sh->B != 1 || sh->N < 1 || sh->N > 65535) return KDA_ERR_SHAPE;
    } else {
        if (sh->N != sh->B || sh->B > 65535) return KDA_ERR_SHAPE;
    }
    if (sh->B * sh->T * sh->H >= (int64_t(1) << 31)) return KDA_ERR_SHAPE;
    if (sh->groups < 0) return KDA_ERR_SHAPE;
    // chunk length: 64 (0 reads as 64) or 32, both served by the 64-token chunk kernels
    if (sh->chunk_size != 0 && sh->chunk_size != 32 && sh->chunk_size != 64) return KDA_ERR_UNSUPPORTED;
    if (sh->groups > 1 && sh->H % sh->groups != 0) return KDA_ERR_SHAPE;
    return KDA_OK;
}

int64_t groups_of(const kda_shape* sh) { return sh->groups > 1 ? sh->groups : 1; }

// FNV-1a hash of everything in the shape that decides the workspace's contents, and of
// whether offsets are given: the provenance stamp kda_fwd leaves and kda_bwd checks.
uint64_t shape_hash(const kda_shape* sh, bool packed) {
    uint64_t h = 1469598103934665603ull;
    auto mix = [&](uint64_t x) {
        for (int i = 0; i < 8; ++i) {
            h ^= (x >> (8 * i)) & 0xffu;
            h *= 1099511628211ull;
        }
    };
    uint32_t sb, lb;
    memcpy(&sb, &sh->scale, 4);
    memcpy(&lb, &sh->lower_bound, 4);
    mix((uint64_t)sh->B); mix((uint64_t)sh->T); mix((uint64_t)sh->H); mix((uint64_t)sh->N);
    mix((uint64_t)groups_of(sh)); mix(sb); mix(lb);
    mix((uint64_t)(sh->chunk_size == 32 ? 32 : 64)); mix(packed ? 1u : 0u);
    return h;
}

Layout layout_of(const kda_shape* sh, bool packed) {
    return make_layout(sh->B, sh->T, sh->H, sh->N, packed, groups_of(sh));
}

// Grid of a persistent per-tile kernel: one CTA (or one two-CTA cluster) per SM,
// never more than tiles.
unsigned persistent_grid(int64_t tiles) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        sms = 148;
    return (unsigned)(tiles < sms ? (tiles > 0 ? tiles : 1) : sms);
}

template <typename K>
kda_status set_smem(K kernel, size_t bytes) {
    return cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes),
                       "cudaFuncSetAttribute");
}

// forward_only: the workspace need only hold the regions the forward writes (status,
// chunk tables, intra-chunk images, S0 and Ut checkpoints: everything before `ds`).
kda_status common_checks(const kda_shape* shape, const int64_t* cu, void* ws, size_t ws_bytes, Layout* lay,
                         bool forward_only = false) {
    const bool packed = cu != nullptr;
    kda_status st = check_shape(shape, packed);
    if (st != KDA_OK) return st;
    *lay = layout_of(shape, packed);
    if (!ws || ws_bytes < (forward_only ? lay->ds : lay->total)) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws) || (packed && (reinterpret_cast<uintptr_t>(cu) & 7u))) return KDA_ERR_ALIGN;
    return KDA_OK;
}

}  // namespace

extern "C" size_t kda_workspace_size(const kda_shape* shape) {
    if (!shape) return 0;
    // the same shape may be used with or without offsets; cover both layouts
    const bool ok_p = check_shape(shape, true) == KDA_OK, ok_f = check_shape(shape, false) == KDA_OK;
    if (!ok_p && !ok_f) return 0;
    const size_t a = ok_p ? layout_of(shape, true).total : 0;
    const size_t b = ok_f ? layout_of(shape, false).total : 0;
    return a > b ? a : b;
}

namespace kda {

// Bytes of the regions the forward alone writes (the forward-only workspace), 0 for an
// invalid shape.
size_t forward_workspace_bytes(const kda_shape* shape, bool packed) {
    if (check_shape(shape, packed) != KDA_OK) return 0;
    return layout_of(shape, packed).ds;
}

// kda_fwd; forward_only: accept a workspace that holds only the forward's regions
// (the backward cannot run on it).
kda_status fwd_entry(const kda_shape* shape, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                     const kda_bf16* g_raw, const kda_bf16* beta_raw, const float* A_log, const float* dt_bias,
                     const float* h0, const int64_t* cu_seqlens, kda_bf16* o, float* hT, void* workspace,
                     size_t workspace_bytes, void* stream, bool forward_only) {
    Layout lay;
    kda_status st = common_checks(shape, cu_seqlens, workspace, workspace_bytes, &lay, forward_only);
    if (st != KDA_OK) return st;
    // with no tokens at all (every sequence empty) the token tensors are empty and may be NULL
    const bool has_tokens = shape->B * shape->T > 0;
    if ((has_tokens && (!q || !k || !v || !g_raw || !beta_raw || !o)) || !A_log || !dt_bias) return KDA_ERR_NULL;
    const void* ptrs[] = {q, k, v, g_raw, beta_raw, A_log, dt_bias, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGN;
    if ((h0 && !aligned16(h0)) || (hT && !aligned16(hT))) return KDA_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int H = (int)shape->H;
    const int64_t T_total = shape->B * shape->T;
    const FwdIntraKernel intra = fwd_intra_kernel(lay.G > 1);
    if ((st = set_smem(intra, fwd_intra_smem_bytes())) != KDA_OK) return st;
    if ((st = set_smem(kda_fwd_scan_kernel, fwd_scan_smem_bytes())) != KDA_OK) return st;

    prof(0, s);
    kda_chunk_table_kernel<<<1, 1024, 0, s>>>(cu_seqlens, shape->N, T_total, cu_seqlens ? 0 : shape->T, ws, lay,
                                              shape_hash(shape, cu_seqlens != nullptr), forward_only ? 0 : 1);
    prof(1, s);
    if (lay.nc_max > 0 && T_total > 0)
        intra<<<persistent_grid(lay.nc_max * H), 512, fwd_intra_smem_bytes(), s>>>(
            q, k, v, g_raw, beta_raw, A_log, dt_bias, H, shape->lower_bound, shape->scale, ws, lay);
    prof(2, s);
    if (shape->N > 0)
        kda_fwd_scan_kernel<<<dim3((unsigned)H, (unsigned)shape->N), 256, fwd_scan_smem_bytes(), s>>>(
            h0, o, hT, H, shape->scale, ws, lay);
    prof(3, s);
    return cuda_status(cudaGetLastError(), "kda_fwd launch");
}

}  // namespace kda

extern "C" kda_status kda_fwd(const kda_shape* shape, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                              const kda_bf16* g_raw, const kda_bf16* beta_raw, const float* A_log,
                              const float* dt_bias, const float* h0, const int64_t* cu_seqlens, kda_bf16* o,
                              float* hT, void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_entry(shape, q, k, v, g_raw, beta_raw, A_log, dt_bias, h0, cu_seqlens, o, hT, workspace,
                     workspace_bytes, stream, false);
}

extern "C" kda_status kda_bwd(const kda_shape* shape, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                              const kda_bf16* g_raw, const kda_bf16* beta_raw, const float* A_log,
                              const float* dt_bias, const float* h0, const int64_t* cu_seqlens, const kda_bf16* do_,
                              const float* dhT, kda_bf16* dq, kda_bf16* dk, kda_bf16* dv, kda_bf16* dg_raw,
                              kda_bf16* dbeta_raw, float* dA_log, float* ddt_bias, float* dh0, void* workspace,
                              size_t workspace_bytes, void* stream) {
    (void)h0;   // the forward's checkpoints in the workspace carry the initial state
    Layout lay;
    kda_status st = common_checks(shape, cu_seqlens, workspace, workspace_bytes, &lay);
    if (st != KDA_OK) return st;
    // with no tokens at all (every sequence empty) the token tensors are empty and may be NULL
    const bool has_tokens = shape->B * shape->T > 0;
    if ((has_tokens && (!q || !k || !v || !g_raw || !beta_raw || !do_ || !dq || !dk || !dv || !dg_raw || !dbeta_raw)) ||
        !A_log || !dt_bias || !dA_log || !ddt_bias)
        return KDA_ERR_NULL;
    const void* ptrs[] = {q, k, v, g_raw, beta_raw, A_log, dt_bias, do_, dq, dk, dv, dg_raw, dbeta_raw, dA_log, ddt_bias};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGN;
    if ((dhT && !aligned16(dhT)) || (dh0 && !aligned16(dh0))) return KDA_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int H = (int)shape->H;
    const float lb = shape->lower_bound, scale = shape->scale;
    if ((st = set_smem(kda_bwd_scan_kernel, bwd_scan_smem_bytes())) != KDA_OK) return st;
    if ((st = set_smem(kda_bwd_state_kernel, bwd_state_smem_bytes())) != KDA_OK) return st;
    const BwdWyKernel wy = bwd_wy_kernel(lay.G > 1);
    const BwdPairKernel pair = bwd_pair_kernel(lay.G > 1);
    if ((st = set_smem(wy, bwd_wy_smem_bytes())) != KDA_OK) return st;
    if ((st = set_smem(pair, bwd_pair_smem_bytes())) != KDA_OK) return st;
    // clusters of two CTAs, two CTAs per SM: all of the unified L1 as shared memory
    if ((st = cuda_status(cudaFuncSetAttribute(pair, cudaFuncAttributePreferredSharedMemoryCarveout,
                                               (int)cudaSharedmemCarveoutMaxShared),
                          "cudaFuncSetAttribute")) != KDA_OK)
        return st;
    const dim3 tiles((unsigned)lay.nc_max, (unsigned)H);
    prof(4, s);
    if (shape->N > 0)
        kda_bwd_scan_kernel<<<dim3((unsigned)H, (unsigned)shape->N), 256, bwd_scan_smem_bytes(), s>>>(
            do_, dhT, dh0, H, ws, lay, shape_hash(shape, cu_seqlens != nullptr));
    prof(5, s);
    if (lay.nc_max > 0)
        kda_bwd_state_kernel<<<persistent_grid(lay.nc_max * H), 512, bwd_state_smem_bytes(), s>>>(do_, H, scale, ws,
                                                                                                  lay);
    prof(6, s);
    if (lay.nc_max > 0)
        wy<<<persistent_grid(lay.nc_max * H), 512, bwd_wy_smem_bytes(), s>>>(k, v, g_raw, beta_raw, A_log, dt_bias, H, lb, dv,
                                                                   ws, lay);
    prof(7, s);
    if (lay.nc_max > 0)
        pair<<<2 * persistent_grid(lay.nc_max * H), 256, bwd_pair_smem_bytes(), s>>>(q, k, g_raw, beta_raw, A_log, dt_bias, H, lb,
                                                                       dq, dk, dg_raw, dbeta_raw, ws, lay);
    const int64_t tokens = shape->B * shape->T;
    if (lay.G > 1 && tokens > 0) {   // grouped value heads: dq, dk summed over each group
        const int64_t rows = tokens * (lay.H / lay.G);   // (token, query/key head) rows of 128 channels
        kda_qk_group_reduce_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(dq, dk, ws, tokens, lay);
    }
    prof(8, s);
    kda_param_reduce_kernel<<<dim3((unsigned)H, (unsigned)kParamGroups), 128, 0, s>>>(H, dA_log, ddt_bias, ws, lay);
    prof(9, s);
    return cuda_status(cudaGetLastError(), "kda_bwd launch");
}

extern "C" const char* kda_last_error(void) { return g_last_error; }

namespace kda {
void set_last_error_text(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }
}  // namespace kda

extern "C" int kda_set_profile_events(void* const* events, int count) {
    g_prof = reinterpret_cast<const cudaEvent_t*>(events);
    g_prof_n = events ? count : 0;
    return KDA_OK;
}

extern "C" kda_status kda_get_device_status(const void* workspace, void* stream) {
    if (!workspace) return KDA_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda_status st = cuda_status(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    if (st != KDA_OK) return st;
    int word = 0;
    st = cuda_status(cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost), "cudaMemcpy");
    if (st != KDA_OK) return st;
    return static_cast<kda_status>(word);
}

extern "C" const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_NULL: return "KDA_ERR_NULL";
        case KDA_ERR_ALIGN: return "KDA_ERR_ALIGN";
        case KDA_ERR_SHAPE: return "KDA_ERR_SHAPE";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_OFFSETS: return "KDA_ERR_OFFSETS";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_STALE_WORKSPACE: return "KDA_ERR_STALE_WORKSPACE";
    }
    return "KDA_ERR_UNKNOWN";
}
