/*
 * kda.h — C ABI of the GB300 (sm_103a) Kimi Delta Attention library.
 *
 * The operation (flashinfer "kda_backward" page, "Supported contract"; FLA
 * chunk_kda call contract on the Kimi-K3 "fused_chunk" page): per sequence n
 * and head h, a value-first fp32 state S in R^{V x K} (K = V = 128) evolves as
 *
 *   q^ = q / sqrt(|q|^2 + 1e-6),  k^ = k / sqrt(|k|^2 + 1e-6)
 *   beta_t = sigmoid(beta_raw_t)
 *   g_t[c] = lower_bound * sigmoid(exp(A_log[h]) * (g_raw_t[c] + dt_bias[h,c]))
 *   S_t = S_{t-1} diag(exp(g_t)) (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T
 *   o_t = scale * S_t q^_t
 *
 * with the decay applied per KEY channel c (the kda-neuron-kernels log, fix
 * T-KDA-02). kda_fwd computes o and the final state; kda_bwd returns the
 * gradients of L = sum_t <o_t, do_t> + <S_T, dhT> w.r.t. q, k, v, g_raw,
 * beta_raw, A_log, dt_bias and the initial state (the list on the flashinfer
 * page).
 *
 * Conventions
 *  - bf16 tensors are passed as raw 16-bit patterns (kda_bf16).
 *  - Token tensors are contiguous [B*T, H, 128] (fixed-length batches, B rows
 *    of T tokens) or [T_total, H, 128] with B = 1 when packed. beta_raw and
 *    dbeta_raw are [B*T, H]. With grouped value heads (kda_shape.groups = G),
 *    q, k, dq, dk are [B*T, H/G, 128] and every other token tensor has H heads.
 *  - A_log, dA_log: [H] fp32. dt_bias, ddt_bias: [H, 128] fp32 (one bias per
 *    key channel of the gate).
 *  - States h0, hT, dhT, dh0: [N, H, V, K] fp32, value-first.
 *  - cu_seqlens: DEVICE pointer to N+1 int64 offsets (0 = cu[0] <= ... <=
 *    cu[N] = T_total) for packed variable-length input; NULL for B fixed
 *    sequences of T tokens (then N = B). Empty sequences are allowed.
 *  - All device pointers must be 16-byte aligned. When B*T = 0 (every sequence
 *    empty) the token tensors are empty and their pointers may be NULL.
 *  - Nullable inputs (h0, dhT) mean zero. Nullable outputs (hT, dh0) are
 *    skipped.
 *  - `stream` is a cudaStream_t. Calls are asynchronous: nothing is
 *    synchronised or allocated inside the launch path.
 *
 * Ownership: the caller owns every buffer, including the workspace. kda_fwd
 * stores its per-chunk intermediates and state checkpoints in the workspace;
 * kda_bwd must receive the same workspace, unchanged, with the same inputs.
 * One workspace must not be used by two calls in flight at the same time.
 *
 * Errors: argument problems are reported synchronously as kda_status codes.
 * Problems found on the device (malformed cu_seqlens, a wait that timed out,
 * a stale workspace) set a status word in the workspace; later kernels of the
 * same call skip their work, and kda_get_device_status() returns the word.
 *
 * Workspace provenance: kda_fwd stamps the workspace with a hash of its shape
 * (B, T, H, N, groups, scale, lower_bound, chunk length, packed or fixed) and,
 * once its last kernel has finished without error, a "forward complete" word.
 * The first kernel of kda_bwd compares both with its own shape; on a mismatch
 * (a workspace from another shape, from no forward at all, or from a forward
 * that failed) it sets KDA_ERR_STALE_WORKSPACE and the backward computes
 * nothing. Only the shape is stamped: the caller still has to pass the same
 * input tensors to both calls.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kda_bf16;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,        /* a required pointer is NULL */
    KDA_ERR_ALIGN = 2,       /* a pointer is not 16-byte aligned */
    KDA_ERR_SHAPE = 3,       /* B, T, H or N out of range / inconsistent */
    KDA_ERR_UNSUPPORTED = 4, /* K or V != 128, lower_bound not in [-5, 0), bad scale */
    KDA_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than required */
    KDA_ERR_OFFSETS = 6,     /* (device) cu_seqlens not 0 .. T_total non-decreasing */
    KDA_ERR_TIMEOUT = 7,     /* (device) a bounded wait inside a kernel gave up */
    KDA_ERR_CUDA = 8,        /* a CUDA launch or attribute call failed */
    KDA_ERR_STALE_WORKSPACE = 9 /* (device) kda_bwd got a workspace that does not hold a
                                   completed kda_fwd of the same shape */
} kda_status;

typedef struct {
    int64_t B;           /* fixed-length batch rows; 1 when packed */
    int64_t T;           /* tokens per row; total tokens when packed */
    int64_t H;           /* heads */
    int64_t N;           /* sequences: B when cu_seqlens is NULL, else len(cu_seqlens) - 1 */
    int32_t K;           /* key dimension, must be 128 */
    int32_t V;           /* value dimension, must be 128 */
    float scale;         /* output scale, finite and > 0 (the pages fix 1/sqrt(128)) */
    float lower_bound;   /* gate lower bound lb, in [-5, 0) (FLA chunk_kda lower_bound) */
    int32_t groups;      /* grouped value heads (the FlashKDA CPU-reference proposal): value
                            heads per query/key head, G >= 1 dividing H (0 is read as 1).
                            H counts value heads; q, k, dq, dk hold H / G heads and value
                            head h reads query/key head h / G; dq, dk are the sums over
                            each group (fixed order). Every other tensor is per value head. */
    int32_t chunk_size;  /* chunk length the caller asks for: 0 or 64 (the default), or 32.
                            The Kimi-K3 fused_chunk validator admits chunk lengths 32 and 64.
                            The chunk length blocks the computation and does not change the
                            function computed, so a request for 32 is served by the 64-token
                            chunk kernels and gives the same results bit for bit. Any other
                            value returns KDA_ERR_UNSUPPORTED. */
} kda_shape;

/* Bytes of workspace kda_fwd and kda_bwd need for this shape (the same buffer
 * serves both; pass at least this many bytes to each). Returns 0 for an
 * invalid shape. */
size_t kda_workspace_size(const kda_shape* shape);

/* Forward. Writes o [B*T, H, 128] bf16 and, if hT != NULL, the final states
 * [N, H, 128, 128] fp32. Fills the workspace with what kda_bwd needs. */
kda_status kda_fwd(const kda_shape* shape,
                   const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                   const kda_bf16* g_raw, const kda_bf16* beta_raw,
                   const float* A_log, const float* dt_bias,
                   const float* h0, const int64_t* cu_seqlens,
                   kda_bf16* o, float* hT,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Backward of the kda_fwd call that filled `workspace`, with the same inputs.
 * do_ is the output adjoint [B*T, H, 128] bf16; dhT the final-state adjoint
 * (NULL = 0). Writes dq, dk [B*T, H/G, 128], dv, dg_raw [B*T, H, 128] bf16, dbeta_raw
 * [B*T, H] bf16, dA_log [H] fp32, ddt_bias [H, 128] fp32 (written, not
 * accumulated) and, if dh0 != NULL, dh0 [N, H, 128, 128] fp32. The parameter
 * gradients are summed over all tokens of all sequences in a fixed order
 * (bitwise reproducible). */
kda_status kda_bwd(const kda_shape* shape,
                   const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                   const kda_bf16* g_raw, const kda_bf16* beta_raw,
                   const float* A_log, const float* dt_bias,
                   const float* h0 /* unused: the forward's checkpoints carry it; may be NULL */,
                   const int64_t* cu_seqlens,
                   const kda_bf16* do_, const float* dhT,
                   kda_bf16* dq, kda_bf16* dk, kda_bf16* dv, kda_bf16* dg_raw,
                   kda_bf16* dbeta_raw, float* dA_log, float* ddt_bias, float* dh0,
                   void* workspace, size_t workspace_bytes, void* stream);

/* One decode step for a batch of requests: the single-token step of the
 * recurrence above, batched over (request, head) pairs (the batched decode
 * entry of the kda-neuron-kernels commit log). For each of the n_req requests
 * and H heads, one token of q, k, v, g_raw [n_req, H, 128] bf16 and beta_raw
 * [n_req, H] bf16 advances the value-first state [n_req, H, 128, 128] fp32
 * IN PLACE and writes o [n_req, H, 128] bf16 (read from the updated state).
 * groups > 1: grouped value heads as in kda_shape.groups (q, k are
 * [n_req, H / groups, 128]; value head h reads query/key head h / groups);
 * 0 or 1: the plain layout.
 * A_log [H] and dt_bias [H, 128] fp32 as in kda_fwd. No workspace; the caller
 * owns every buffer. The result is that of kda_fwd over sequences of one token
 * with h0 = the state before and hT = the state after.
 * Errors: n_req < 0, H <= 0, n_req * H >= 2^31, groups < 0 or groups > 1 not
 * dividing H -> KDA_ERR_SHAPE; scale not
 * finite and > 0, or lower_bound outside [-5, 0) -> KDA_ERR_UNSUPPORTED; a NULL
 * pointer (n_req > 0) -> KDA_ERR_NULL; a pointer not 16-byte aligned ->
 * KDA_ERR_ALIGN; a failed launch -> KDA_ERR_CUDA (text in kda_last_error()).
 * n_req = 0 does nothing. */
kda_status kda_decode(long long n_req, long long H, long long groups, float scale, float lower_bound,
                      const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                      const kda_bf16* g_raw, const kda_bf16* beta_raw,
                      const float* A_log, const float* dt_bias,
                      float* state, kda_bf16* o, void* stream);

/* Synchronises `stream` and returns the device status word of `workspace`
 * (KDA_OK, KDA_ERR_OFFSETS, KDA_ERR_TIMEOUT or KDA_ERR_STALE_WORKSPACE), or
 * KDA_ERR_CUDA if the stream reported an error. Clears nothing. */
kda_status kda_get_device_status(const void* workspace, void* stream);

/* Profiling hook. When `events` is non-NULL (an array of `count` cudaEvent_t
 * created by the caller), kda_fwd records events[0..3] and kda_bwd
 * events[4..9] on the call's stream around its kernels:
 *   [0,1) status clear + chunk table   [1,2) intra-chunk   [2,3) forward scan
 *   [4,5) backward scan  [5,6) state products  [6,7) WY backward
 *   [7,8) pair/gate backward  [8,9) parameter reduction
 * (events[3] and events[9] mark the end of each call). Process-wide setting,
 * not thread-safe; pass NULL to switch it off. Returns KDA_OK. */
int kda_set_profile_events(void* const* events, int count);

/* Bytes of the scratch array compiled into the library for
 * kda_fwd_static_scratch (64 MiB). */
#define KDA_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* kda_fwd for callers that cannot allocate device memory. The pages have no
 * counterpart of this entry point; it exists for the library's users.
 *
 * Some callers may not call cudaMalloc or any allocator: code running inside
 * another runtime's plugin or custom-op interface, where the host program owns
 * every device allocation, and serving loops that must not allocate, because
 * an allocation can synchronise the device and stall other work. This entry
 * point takes the same arguments as kda_fwd without the workspace: it uses a
 * scratch array of KDA_STATIC_SCRATCH_BYTES compiled into the library, which
 * every GPU that loads the library's code holds until the process exits.
 * It calls no allocating routine.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture on that device.
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents (what must start at zero is cleared by each call). Calls whose
 *    work overlaps on the GPU (other streams, other host threads) race on it:
 *    serialise them.
 *  - Only the forward runs, so only the workspace regions the forward writes
 *    must fit: about 160 (chunk of 64 tokens, head) tiles, e.g. T = 2048 with
 *    H = 4. Larger shapes return KDA_ERR_WORKSPACE, and kda_last_error()
 *    states both sizes.
 *  - Forward only: the intermediates it keeps are not available to kda_bwd.
 *  - Problems found on the device (malformed cu_seqlens, a timed-out wait) go
 *    to the status word of the scratch array, not to a workspace of the
 *    caller's: read them with kda_static_scratch_device_status().
 *  - The cached address is not renewed: after cudaDeviceReset() on a device,
 *    this entry point must not be called again on it in the same process.
 * Host-side errors are those of kda_fwd. */
kda_status kda_fwd_static_scratch(const kda_shape* shape,
                                  const kda_bf16* q, const kda_bf16* k, const kda_bf16* v,
                                  const kda_bf16* g_raw, const kda_bf16* beta_raw,
                                  const float* A_log, const float* dt_bias,
                                  const float* h0, const int64_t* cu_seqlens,
                                  kda_bf16* o, float* hT, void* stream);

/* Synchronises `stream` and returns the device status word of the scratch array
 * that kda_fwd_static_scratch uses on the current device (KDA_OK,
 * KDA_ERR_OFFSETS or KDA_ERR_TIMEOUT from the last call there), or KDA_ERR_CUDA.
 * No counterpart on the pages either. */
kda_status kda_static_scratch_device_status(void* stream);

/* Text of the last CUDA error an entry point of the calling thread turned
 * into KDA_ERR_CUDA ("" if none). Static per-thread buffer. */
const char* kda_last_error(void);

/* Human-readable name of a status code (static string). */
const char* kda_status_string(kda_status s);

/* Diagnostics: one CTA computes D[128 x N] = A[128 x Kd] * B[N x Kd]^T with
 * tcgen05 kind::tf32 (operands rounded to tf32), both operands stored in
 * shared memory K-major with the 128-byte swizzle the kernels use (a_mn and
 * b_mn must be 0: tf32 operands are K-major only; anything else returns
 * KDA_ERR_UNSUPPORTED). D holds 2*128*N floats: the product, then
 * (2 * product + row index) after a round trip through tcgen05.st /
 * tcgen05.ld. A, B, D are device pointers, row-major. N in {16, 32, ..., 256},
 * Kd in {32, 64, 96, 128} (else KDA_ERR_SHAPE). Used by the tests to check
 * the descriptors and the TMEM data path. */
int kda_diag_umma_selftest(int a_mn, int b_mn, int N, int Kd, const float* A, const float* B,
                           float* D, void* stream);

/* Diagnostics: launches one CTA that waits on an mbarrier nothing completes,
 * gives up after limit_ns (1 .. 1e9 ns), and sets KDA_ERR_TIMEOUT in the
 * status word of `workspace` (its first 4 bytes, device memory) exactly as a
 * timed-out wait inside kda_fwd / kda_bwd would. Read it with
 * kda_get_device_status(). Used by the tests of the failure path; the
 * context stays usable afterwards. */
int kda_diag_wait_timeout(unsigned long long limit_ns, void* workspace, void* stream);

/* Diagnostics: for each of the n floats in `in` (device memory) writes the
 * library's own tf32 rounding to `out` and the hardware conversion
 * cvt.rna.tf32.f32 (round to nearest, ties away from zero) to `ref` (device
 * memory, n floats each, caller-owned). The kernels round tf32 operands with
 * integer operations (add half a tf32 unit in the last place to the magnitude
 * bits unless the value is a NaN, clear the 13 bits below tf32); the tests use
 * this entry point to check that it equals the hardware conversion bit for
 * bit on every input. n < 0 gives
 * KDA_ERR_SHAPE, a null pointer (n > 0) KDA_ERR_NULL. */
int kda_diag_tf32_round(const float* in, float* out, float* ref, long long n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
