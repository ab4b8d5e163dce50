// Forward pass for callers that cannot allocate device memory.
//
// Some callers of this library may not call cudaMalloc (or any allocator):
// code that runs inside another runtime's plugin or custom-op interface where
// the host program owns every device allocation, and serving loops that must
// not allocate (an allocation can synchronise the device and stall other
// streams). kda_fwd needs a caller-provided workspace; this entry point
// instead uses a fixed scratch array compiled into the library, so the caller
// passes only its inputs and outputs.
//
// The scratch is a file-scope __device__ array of KDA_STATIC_SCRATCH_BYTES.
// Every GPU on which this library's code is loaded holds it until the process
// exits. In host code the array's name is only a host-side stand-in, so the
// device address is looked up once per device with cudaGetSymbolAddress and
// cached.
#include <cstdio>
#include <mutex>
#include "kda_internal.cuh"

namespace kda {
void set_last_error_text(const char* msg);
size_t forward_workspace_bytes(const kda_shape* shape, bool packed);
kda_status fwd_entry(const kda_shape* shape, const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                     const kda_bf16* g_raw, const kda_bf16* beta_raw, const float* A_log, const float* dt_bias,
                     const float* h0, const int64_t* cu_seqlens, kda_bf16* o, float* hT, void* workspace,
                     size_t workspace_bytes, void* stream, bool forward_only);
}

namespace {

constexpr size_t kStaticScratchBytes = (size_t)KDA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up on
// the first call per device and kept for the life of the process (a device reset,
// which reloads the library's module, is not supported afterwards).
kda_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        kda::set_last_error_text("kda_fwd_static_scratch: cudaGetDevice failed");
        return KDA_ERR_CUDA;
    }
    if (dev >= kMaxDevices) {
        kda::set_last_error_text("kda_fwd_static_scratch: device index beyond the supported 64");
        return KDA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) {
            kda::set_last_error_text("kda_fwd_static_scratch: cudaGetSymbolAddress failed");
            return KDA_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_fwd_static_scratch(const kda_shape* shape, const kda_bf16* q, const kda_bf16* k,
                                             const kda_bf16* v, const kda_bf16* g_raw, const kda_bf16* beta_raw,
                                             const float* A_log, const float* dt_bias, const float* h0,
                                             const int64_t* cu_seqlens, kda_bf16* o, float* hT, void* stream) {
    if (!shape) return KDA_ERR_NULL;
    // the forward alone runs here: it needs only the workspace regions it writes
    const size_t need = kda::forward_workspace_bytes(shape, cu_seqlens != nullptr);
    if (need == 0) return KDA_ERR_SHAPE;
    if (need > kStaticScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "kda_fwd_static_scratch: this shape needs %zu bytes of scratch; the static scratch holds %zu",
                 need, kStaticScratchBytes);
        kda::set_last_error_text(msg);
        return KDA_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    const kda_status st = scratch_address(&scratch);
    if (st != KDA_OK) return st;
    // the forward clears the status word and rebuilds every table it reads; no
    // other part of the scratch needs to start at zero.
    return kda::fwd_entry(shape, q, k, v, g_raw, beta_raw, A_log, dt_bias, h0, cu_seqlens, o, hT, scratch,
                          kStaticScratchBytes, stream, true);
}

// The device status word of the last kda_fwd_static_scratch call on the current device
// (malformed offsets or a timed-out wait found on the device are reported only there:
// the caller never sees the scratch array's address).
extern "C" kda_status kda_static_scratch_device_status(void* stream) {
    void* scratch = nullptr;
    const kda_status st = scratch_address(&scratch);
    if (st != KDA_OK) return st;
    return kda_get_device_status(scratch, stream);
}
