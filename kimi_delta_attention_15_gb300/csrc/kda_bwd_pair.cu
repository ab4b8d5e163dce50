// Backward, last per-chunk stage, per (chunk, head) tile. Gathers every adjoint of
// q^, k^ and of the in-chunk cumulative log-decay G, then applies the reverse
// cumulative sum (g_t = G_t - G_{t-1}) and the chains of the gate, the beta sigmoid
// and the L2 norms:
//   pair terms  B_ij = sum_c k^_ic k^_jc e^{G_ic-G_jc},  Aqk_ij = sum_c q^_ic k^_jc e^{G_ic-G_jc}
//     with dB (WY kernel) and dAqk (state-products kernel), for column block J:
//     a = dM[:,J] Kt_J,  b = dM[:,J]^T Xt_J   (Xt_J = x^ e^{G-G_eJ}, Kt_J = k^_J e^{G_eJ-G_J})
//     dx += e^{G-G_eJ} a,  dk_J += e^{G_eJ-G_J} b,  dG += Xt_J a,  dG_J -= Kt_J b
//     (products about fp32 accurate: tf32 high parts plus bf16 cross terms,
//      mma_sync.cuh; both dG terms multiply the
//      same factors k^, E-, E+ and f_IJ, rounded to fp32 at most once apart, so the
//      pairs inside [t, L) cancel in the reverse cumulative sum to fp32 accuracy);
//   dq^ += dQbar Gamma, dk^ += dKt Gamma + dKbar e^{G_L-G},
//   dG  += dQbar Q^Gamma + dKt K^Gamma - dKbar Kbar,
//   dG_L = sum_i dKbar_i Kbar_i + dgam exp(G_L).
// dg_t = sum_{i>=t} dG_i + dG_L is assembled as
//   sum_{i>=t} (dG_i without the Kbar term) + sum_{i<t} dKbar_i Kbar_i + dgam exp(G_L)
// which is the same sum without the cancellation of the Kbar terms.
// Then du = dg lb s (1 - s), dg_raw = du exp(A_log), and the per-chunk
// partial sums of ddt_bias and dA_log go to the workspace.
//
// Every term above is per key channel except the row norms of q and k and the row
// dot products of the L2-norm chains. A cluster of two CTAs takes each tile, CTA r
// the key channels 64r .. 64r+63; the two exchange those per-row partial sums
// through distributed shared memory: st.async writes into the peer, counted in bytes on
// the peer's mbarrier, so that no fence waits for this CTA's own global traffic. Half the channels need half the shared memory
// (about 107 KB), so two CTAs share an SM and the memory phases of one overlap the
// arithmetic of the other. Persistent over tiles; the raw q, k, g_raw rows of the
// cluster's next tile are staged by cp.async in the dAqk and dB tiles, which are
// free from the write-back of the adjoints to the end of the tile.
// Grouped value heads (G value heads per query/key head): the q, k rows come from
// query/key head h / G, and dq, dk leave as each value head's fp32 share, summed per
// group by kda_qk_group_reduce_kernel (end of this file).
#include "kda_internal.cuh"
#include "kda_prep.cuh"
#include "mma_sync.cuh"
#include "umma.cuh"

namespace kda {

namespace {
constexpr int CH = D / 2;   // key channels per CTA
constexpr int kPairWarps = 8;
constexpr int kPairThreads = kPairWarps * 32;
static_assert(CH == C, "the [64][64] tiles share one layout");

// dB and dAqk: [64][64] fp32, rows of 64 floats with the column index XOR-ed by a
// function of the row, so that the mma fragment loads in both orientations (row by
// lane / 4 and column by lane % 4, or the transpose) are free of bank conflicts.
// Aligned groups of four columns stay contiguous (16-byte copies keep working).
__device__ __forceinline__ int sw(int r, int c) { return r * CH + (c ^ (((r & 3) << 3) | (r & 4))); }
// [64][64] fp32 channel tiles: rows padded to 72 floats (plain addressing with constant
// offsets). A row stride of 8 banks keeps the two access patterns these tiles see free of
// bank conflicts: mma fragments with the row by lane % 4 and the column by lane / 4, and
// 8-byte element pairs with the row by lane / 4 and the column pair by lane % 4.
constexpr int PCH = CH + 8;
__device__ __forceinline__ int pidx(int r, int c) { return r * PCH + c; }

// block-pair factors f_IJ of the lower triangle J <= I, at fidx(I, J)
__device__ __forceinline__ int fidx(int I, int J) { return I * (I + 1) / 2 + J; }
struct PairFactors {
    float F[NSUB * (NSUB + 1) / 2][CH];
    float Pb[NSUB][CH];
    float Sf[NSUB][CH];
    float Db[NSUB][CH];
    float gl[CH];
};

struct PairSmem {
    float qe[C * PCH];   // q^ E-          -> dq^
    float ke[C * PCH];   // k^ E-          -> dk^
    float kp[C * PCH];   // alpha, k^ E+   -> dG'
    float em[C * PCH];   // E-             -> dKbar Kbar, then its exclusive prefix over rows
    float dB[C * C];    // dB; from the write-back on: dg scratch (4 KB), staged g_raw rows
    float dA[C * C];    // dAqk; from the write-back on: staged q and k rows
    PairFactors fa;
    float beta[C], inq[C], ink[C];
    float xn[2][2][C];  // partial squared norms per row: [channel half][q, k][row]
    float xd[2][2][C];  // partial dot products of the L2-norm chains, same layout
    alignas(16) float dtb[CH];
    float red[kPairWarps];
    float go;
    int bad;            // a partial-sum wait timed out: later waits are skipped
    uint16_t braw[C];
    alignas(8) uint64_t mb_xn, mb_xd;   // the peer's 512 bytes of xn, of xd (one phase per tile)
};
static_assert(sizeof(PairSmem) <= 113 * 1024, "two CTAs per SM");

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// v to the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ void st_cluster(const float* local, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
// v to this CTA's and to the peer's copy of a location
__device__ __forceinline__ void st_both(float* local, uint32_t peer, float v) {
    *local = v;
    st_cluster(local, peer, v);
}

// v into the same shared-memory location of CTA `rank`, counted as 4 bytes on that CTA's
// mbarrier at the location of `bar`
__device__ __forceinline__ void st_async_peer(const float* local, const uint64_t* bar, uint32_t rank, float v) {
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra),
                 "r"(__float_as_uint(v)), "r"(rb)
                 : "memory");
}
// one test of a phase of an mbarrier completed by the peer's writes; acquire at cluster
// scope, so that those writes are visible afterwards
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// the rest of a bounded wait (kWaitLimitNs), out of line: the tile loop keeps its registers
__device__ __noinline__ bool mbar_wait_cluster_slow(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_test_cluster(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    return mbar_test_cluster(a, parity) || mbar_wait_cluster_slow(a, parity);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
}  // namespace

size_t bwd_pair_smem_bytes() { return sizeof(PairSmem); }

// kGrouped: q, k, dq, dk hold H / G heads (grouped value heads) and the kernel writes each
// value head's fp32 share of dq, dk to the workspace; the plain layout is its own
// instantiation, writing bf16 dq, dk directly.
template <bool kGrouped>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 2)
    kda_bwd_pair_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                        const uint16_t* __restrict__ g_raw, const uint16_t* __restrict__ beta_raw,
                        const float* __restrict__ A_log, const float* __restrict__ dt_bias, int H, float lb,
                        uint16_t* __restrict__ dq, uint16_t* __restrict__ dk, uint16_t* __restrict__ dg_raw,
                        uint16_t* __restrict__ dbeta_raw, uint8_t* __restrict__ ws, Layout lay) {
    extern __shared__ uint8_t smem_raw[];
    PairSmem& s = *reinterpret_cast<PairSmem*>(smem_raw);
    const uint32_t half = cluster_rank(), peer = half ^ 1u;
    const int cb = (int)half * CH;   // first key channel of this CTA
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    constexpr uint32_t kAll = 0xffffffffu;

    // Both CTAs of the cluster run or neither: rank 0 reads the status word and passes
    // its decision on. The first barrier also makes sure both CTAs have started, and
    // their mbarriers are initialised, before either writes into the other's shared
    // memory; every later step is taken by both CTAs alike (same tiles, same exits), so
    // every cluster barrier is met by both and every partial sum one CTA waits for is
    // sent by the other. A CTA receives its peer's partial sums of a tile only after the
    // peer has read its own of the tile before (each exchange is answered by the next
    // one), so one buffer of each suffices.
    if (tid == 0) {
        mbar_init(&s.mb_xn, 1);
        mbar_init(&s.mb_xd, 1);
        s.bad = 0;
        fence_mbar_init();
    }
    cluster_arrive();
    cluster_wait();
    if (half == 0 && tid == 0) st_both(&s.go, peer, read_status(ws) == 0 ? 1.0f : 0.0f);
    cluster_arrive();
    cluster_wait();
    if (s.go == 0.0f) return;

    const ChunkInfo* chunks = reinterpret_cast<const ChunkInfo*>(ws + lay.chunks);
    const int ntiles = (int)lay.nc_max * H;
    const int step = (int)(gridDim.x >> 1);
    const int G = kGrouped ? (int)lay.G : 1, Hqk = H / G;   // q, k, dq, dk have Hqk heads
    // empty chunk records only follow the last real chunk: the first one ends the work
    int tile_i = (int)(blockIdx.x >> 1);
    ChunkInfo ci = tile_i < ntiles ? chunks[tile_i / H] : ChunkInfo{0, 0, 0, 0};
    if (ci.L <= 0) return;
    uint16_t* const stq = reinterpret_cast<uint16_t*>(s.dA);   // staged rows, [64][64] bf16 each
    uint16_t* const stk = stq + C * CH;
    uint16_t* const stg = reinterpret_cast<uint16_t*>(s.dB + 1024);
    float* const scr = s.dB;                                     // [4][RG][64] dg scratch
    uint16_t* const stgc = reinterpret_cast<uint16_t*>(s.qe);   // the tile's raw gate rows, in the gate chain
    float alog_next = 0.0f;
    uint16_t braw_next = 0;
    // this CTA's channels of the raw rows of tile t_i (record cn); rows past the chunk read as zero
    auto stage_tile = [&](int t_i, const ChunkInfo& cn) {
        const int hn = t_i % H, hq = hn / G;   // value head, its query/key head
        for (int seg = tid; seg < 3 * C * (CH / 8); seg += kPairThreads) {
            const int which = seg >> 9, rem = seg & 511, r = rem >> 3, c8 = (rem & 7) * 8;
            const uint16_t* src = which == 0 ? q : which == 1 ? k : g_raw;
            const bool valid = r < cn.L;
            // q, k belong to query/key head hq (grouped value heads), g_raw to value head hn
            const int hs = which < 2 ? hq : hn, Hs = which < 2 ? Hqk : H;
            src += ((size_t)(cn.t0 + (valid ? r : 0)) * Hs + hs) * D + cb + c8;
            uint16_t* dst = (which == 0 ? stq : which == 1 ? stk : stg) + r * CH + c8;
            cp_async16_zfill(dst, src, valid);
        }
        if (tid < CH / 4) cp_async16(s.dtb + 4 * tid, dt_bias + (size_t)hn * D + cb + 4 * tid);
        cp_async_commit();
        alog_next = A_log[hn];
        if (tid < C) braw_next = tid < cn.L ? beta_raw[(size_t)(cn.t0 + tid) * H + hn] : (uint16_t)0;
    };
    stage_tile(tile_i, ci);
    float alog = alog_next;
    uint16_t braw = braw_next;
    uint32_t par = 0;   // phase parity of mb_xn and mb_xd for this tile
    // after a __syncthreads: wait for the peer's partial sums (skipped once a wait has
    // timed out, which is reported in the status word)
    auto wait_peer = [&](uint64_t* bar) {
        if (s.bad == 0 && !mbar_wait_cluster(bar, par)) {
            s.bad = 1;
            raise_status(ws, KDA_ERR_TIMEOUT);
        }
    };
    while (true) {
    const int nxt = tile_i + step;
    const ChunkInfo cn = nxt < ntiles ? chunks[nxt / H] : ChunkInfo{0, 0, 0, 0};
    const int h = tile_i % H;
    const int L = ci.L, t0 = ci.t0;
    const size_t tile = (size_t)tile_i;
    const uint8_t* bg = ws + lay.bg + tile * BgOff::BYTES;
    const uint8_t* wy = ws + lay.wy + tile * WyOff::BYTES;
    const float a_h = __expf(alog);

    if (tid < C) s.braw[tid] = braw;
    if (tid == 0) {   // this tile's phase of both exchanges: 2 x 64 floats from the peer each
        mbar_arrive_expect_tx(&s.mb_xn, 2 * C * 4);
        mbar_arrive_expect_tx(&s.mb_xd, 2 * C * 4);
    }
    cp_async_wait_all();
    __syncthreads();
    // ---- rows: a half-warp per row, lane l the channels cb + 4(l % 16) .. +3 of row
    // 16b + 2w + l / 16 (b = 0 .. 3)
    constexpr int RB = C / (2 * kPairWarps);
    const int hl = lane >> 4, c4 = 4 * (lane & 15);
    uint2 wq[RB], wk[RB], wg[RB];
#pragma unroll
    for (int b = 0; b < RB; ++b) {
        const int r = 16 * b + 2 * warp + hl;
        wq[b] = *reinterpret_cast<const uint2*>(stq + r * CH + c4);
        wk[b] = *reinterpret_cast<const uint2*>(stk + r * CH + c4);
        wg[b] = *reinterpret_cast<const uint2*>(stg + r * CH + c4);
    }
    const float4 dt4 = *reinterpret_cast<const float4*>(s.dtb + c4);
    __syncthreads();   // the staged rows are read: dB and dAqk are reloaded over them
    {
        const float* gB = reinterpret_cast<const float*>(wy + WyOff::DB);
        const float* gA = reinterpret_cast<const float*>(bg + BgOff::DAQK);
        for (int i = tid; i < 2 * C * (C / 4); i += kPairThreads) {
            const int m = i >> 10, r = (i >> 4) & (C - 1), j = (i & 15) * 4;
            cp_async16((m ? s.dA : s.dB) + sw(r, j), (m ? gA : gB) + r * C + j);
        }
        cp_async_commit();
    }
    // each warp of the products owns rows 16rb + {gid, gid+8}, columns chw + 8nt + 2tig + {0,1}
    const int rb = warp & 3, chw = (warp >> 2) * 32;
    constexpr int NT = 4;   // n-tiles of 8 columns per warp
    const float* gdQ = reinterpret_cast<const float*>(bg + BgOff::DQB) + cb;
    const float* gdKb = reinterpret_cast<const float*>(bg + BgOff::DKB) + cb;
    const float* gdKt = reinterpret_cast<const float*>(wy + WyOff::DKT) + cb;
    // operands of the elementwise terms (dQbar, dKt) of this thread's elements: loaded
    // now, so that their latency hides under the row preparation
    float2 eQ[NT][2], eKt[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int row = rb * SUB + gid + hh * 8, col = chw + nt * 8 + tig * 2;
            eQ[nt][hh] = *reinterpret_cast<const float2*>(gdQ + row * D + col);
            eKt[nt][hh] = *reinterpret_cast<const float2*>(gdKt + row * D + col);
        }

    // ---- row preparation. Squared norms in the fixed order of the other chunk kernels:
    // a fused chain over each lane's 4 channels, a butterfly over the 16 lanes of the
    // row (this half of the channels), then the sum of the two halves' partials
    auto un4 = [](uint2 w, float (&x)[4]) {
        x[0] = bf_lo(w.x); x[1] = bf_hi(w.x); x[2] = bf_lo(w.y); x[3] = bf_hi(w.y);
    };
    {
        float sq[RB], sk[RB];
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            float qv[4], kv[4];
            un4(wq[b], qv); un4(wk[b], kv);
            sq[b] = sq4(qv[0], qv[1], qv[2], qv[3]);
            sk[b] = sq4(kv[0], kv[1], kv[2], kv[3]);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
#pragma unroll
            for (int b = 0; b < RB; ++b) {
                sq[b] += __shfl_xor_sync(kAll, sq[b], o);
                sk[b] += __shfl_xor_sync(kAll, sk[b], o);
            }
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            const int r = 16 * b + 2 * warp + hl;
            if ((lane & 15) < 2) {
                float* x = &s.xn[half][lane & 15][r];
                const float v = (lane & 15) == 0 ? sq[b] : sk[b];
                *x = v;
                st_async_peer(x, &s.mb_xn, peer, v);
            }
        }
    }
    // gates and beta need no norm: computed while the peer's partials arrive
    {
        const float dtv[4] = {dt4.x, dt4.y, dt4.z, dt4.w};
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            const int r = 16 * b + 2 * warp + hl;
            float gr[4], al[4] = {1.0f, 1.0f, 1.0f, 1.0f};
            un4(wg[b], gr);
            if (r < L) {
#pragma unroll
                for (int e = 0; e < 4; ++e) al[e] = __expf(lb * sigmoidf(a_h * (gr[e] + dtv[e])));
            }
            *reinterpret_cast<float4*>(s.kp + pidx(r, c4)) = make_float4(al[0], al[1], al[2], al[3]);
            if ((lane & 15) == 0) s.beta[r] = r < L ? sigmoidf(bf2f(s.braw[r])) : 0.0f;
        }
    }
    __syncthreads();
    wait_peer(&s.mb_xn);
#pragma unroll
    for (int b = 0; b < RB; ++b) {
        const int r = 16 * b + 2 * warp + hl;
        const float iq = rsqrtf(s.xn[0][0][r] + s.xn[1][0][r] + 1e-6f);
        const float ik = rsqrtf(s.xn[0][1][r] + s.xn[1][1][r] + 1e-6f);
        float qv[4], kv[4];
        un4(wq[b], qv); un4(wk[b], kv);
        *reinterpret_cast<float4*>(s.qe + pidx(r, c4)) = make_float4(qv[0] * iq, qv[1] * iq, qv[2] * iq, qv[3] * iq);
        *reinterpret_cast<float4*>(s.ke + pidx(r, c4)) = make_float4(kv[0] * ik, kv[1] * ik, kv[2] * ik, kv[3] * ik);
        if ((lane & 15) == 0) {
            s.inq[r] = iq;
            s.ink[r] = ik;
        }
    }
    cp_async_wait_all();
    __syncthreads();
    // block products: thread (I, c) walks the 16 rows of block I in channel c
    {
        const int c = tid & (CH - 1), I = tid >> 6;
        float al[SUB], e_m[SUB], e_p[SUB];
#pragma unroll
        for (int i = 0; i < SUB; ++i) al[i] = s.kp[pidx(I * SUB + i, c)];
        float pre = 1.0f;
#pragma unroll
        for (int i = 0; i < SUB; ++i) { pre *= al[i]; e_m[i] = pre; }
        float suf = 1.0f;
#pragma unroll
        for (int i = SUB - 1; i >= 0; --i) { e_p[i] = suf; suf *= al[i]; }
        s.fa.Db[I][c] = pre;
#pragma unroll
        for (int i = 0; i < SUB; ++i) {
            const int a = pidx(I * SUB + i, c);
            const float kh = s.ke[a];
            s.ke[a] = kh * e_m[i];
            s.kp[a] = kh * e_p[i];
            s.qe[a] = s.qe[a] * e_m[i];
            s.em[a] = e_m[i];
        }
    }
    __syncthreads();
    if (tid < CH) {   // block factors of channel tid
        const int c = tid;
        const float d0 = s.fa.Db[0][c], d1 = s.fa.Db[1][c], d2 = s.fa.Db[2][c], d3 = s.fa.Db[3][c];
        s.fa.Pb[0][c] = 1.0f; s.fa.Pb[1][c] = d0; s.fa.Pb[2][c] = d0 * d1; s.fa.Pb[3][c] = d0 * d1 * d2;
        s.fa.gl[c] = d0 * d1 * d2 * d3;
        s.fa.Sf[3][c] = 1.0f; s.fa.Sf[2][c] = d3; s.fa.Sf[1][c] = d2 * d3; s.fa.Sf[0][c] = d1 * d2 * d3;
        s.fa.F[fidx(0, 0)][c] = 1.0f / d0; s.fa.F[fidx(1, 1)][c] = 1.0f / d1;
        s.fa.F[fidx(2, 2)][c] = 1.0f / d2; s.fa.F[fidx(3, 3)][c] = 1.0f / d3;
        s.fa.F[fidx(1, 0)][c] = 1.0f; s.fa.F[fidx(2, 1)][c] = 1.0f; s.fa.F[fidx(3, 2)][c] = 1.0f;
        s.fa.F[fidx(2, 0)][c] = d1; s.fa.F[fidx(3, 1)][c] = d2; s.fa.F[fidx(3, 0)][c] = d1 * d2;
    }
    __syncthreads();

    // (c) elementwise terms of Q^*Gamma and K^*Gamma start the accumulators (the Kbar terms
    // follow the pair products, from an L2-warm reload of dKbar)
    float adq[NT][4], adk[NT][4], adg[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int row = rb * SUB + gid + hh * 8, col = chw + nt * 8 + tig * 2, a = pidx(row, col);
            const float2 pb = *reinterpret_cast<const float2*>(&s.fa.Pb[rb][col]);
            const float2 emv = *reinterpret_cast<const float2*>(s.em + a);
            const float2 qev = *reinterpret_cast<const float2*>(s.qe + a);
            const float2 kev = *reinterpret_cast<const float2*>(s.ke + a);
            const float pbv[2] = {pb.x, pb.y}, emx[2] = {emv.x, emv.y}, qex[2] = {qev.x, qev.y},
                        kex[2] = {kev.x, kev.y};
            const float dQv[2] = {eQ[nt][hh].x, eQ[nt][hh].y}, dKtv[2] = {eKt[nt][hh].x, eKt[nt][hh].y};
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int e = hh * 2 + e2;
                const float gam = emx[e2] * pbv[e2];
                const float qb = qex[e2] * pbv[e2], kt = kex[e2] * pbv[e2];
                adq[nt][e] = dQv[e2] * gam;
                adk[nt][e] = dKtv[e2] * gam;
                adg[nt][e] = dQv[e2] * qb + dKtv[e2] * kt;
            }
        }

    // (a) row side: rows of block I = rb, column blocks J <= I. The decay factor f_IJ of
    // each column block is folded into the shared B operand (k^ E+ of block J, times f_IJ
    // per channel), so the products with dB and with dAqk accumulate over all J and the
    // epilogue, with E- of the rows, runs once
    {
        const int I = rb;
        const int r0 = I * SUB + gid, r1 = r0 + 8;
        float accB[NT][4], accA[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) accB[nt][e] = accA[nt][e] = 0.0f;
        for (int J = 0; J <= I; ++J) {
            const float* f = s.fa.F[fidx(I, J)];
            float fc[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) fc[nt] = f[chw + nt * 8 + gid];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int j0 = J * SUB + kk * 8 + tig, j1 = j0 + 4;
                const Frag4x fb = frag4x(s.dB[sw(r0, j0)], s.dB[sw(r1, j0)], s.dB[sw(r0, j1)], s.dB[sw(r1, j1)]);
                const Frag4x fa = frag4x(s.dA[sw(r0, j0)], s.dA[sw(r1, j0)], s.dA[sw(r0, j1)], s.dA[sw(r1, j1)]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int c = chw + nt * 8 + gid;
                    const Frag2x kb = frag2x(s.kp[pidx(j0, c)] * fc[nt], s.kp[pidx(j1, c)] * fc[nt]);
                    mma2x(accB[nt], fb, kb);
                    mma2x(accA[nt], fa, kb);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = I * SUB + gid + hh * 8, col = chw + nt * 8 + tig * 2, a = pidx(row, col);
                const float2 emv = *reinterpret_cast<const float2*>(s.em + a);
                const float2 kev = *reinterpret_cast<const float2*>(s.ke + a);
                const float2 qev = *reinterpret_cast<const float2*>(s.qe + a);
                const float emx[2] = {emv.x, emv.y}, kex[2] = {kev.x, kev.y}, qex[2] = {qev.x, qev.y};
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int e = hh * 2 + e2;
                    adk[nt][e] += emx[e2] * accB[nt][e];
                    adq[nt][e] += emx[e2] * accA[nt][e];
                    adg[nt][e] += kex[e2] * accB[nt][e];
                    adg[nt][e] += qex[e2] * accA[nt][e];
                }
            }
    }
    float pk[NT][4];   // dKbar Kbar of this thread's elements
    // (b) column side: rows j of block J = rb, row blocks I >= J. E+ of those rows is
    // D_J / E- (it enters only dk^, no cancelling term)
    {
        const int J = rb;
        float acc[NT][4], acc2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = acc2[nt][e] = 0.0f;
        for (int I = J; I < NSUB; ++I) {
            const float* f = s.fa.F[fidx(I, J)];
            float fc[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) fc[nt] = f[chw + nt * 8 + gid];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int i0 = I * SUB + kk * 8 + tig, i1 = i0 + 4;
                const int c0 = J * SUB + gid, c1 = c0 + 8;
                const Frag4x ab = frag4x(s.dB[sw(i0, c0)], s.dB[sw(i0, c1)], s.dB[sw(i1, c0)], s.dB[sw(i1, c1)]);
                const Frag4x aa = frag4x(s.dA[sw(i0, c0)], s.dA[sw(i0, c1)], s.dA[sw(i1, c0)], s.dA[sw(i1, c1)]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int c = chw + nt * 8 + gid;
                    mma2x(acc[nt], ab, frag2x(s.ke[pidx(i0, c)] * fc[nt], s.ke[pidx(i1, c)] * fc[nt]));
                    mma2x(acc2[nt], aa, frag2x(s.qe[pidx(i0, c)] * fc[nt], s.qe[pidx(i1, c)] * fc[nt]));
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] += acc2[nt][e];
        // the column-side epilogue and the elementwise Kbar terms act on the same elements
        // (rows of block J = rb): E+ = D_J / E- once per element
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = J * SUB + gid + hh * 8, col = chw + nt * 8 + tig * 2, a = pidx(row, col);
                const float2 dKb2 = *reinterpret_cast<const float2*>(gdKb + row * D + col);
                const float2 sf = *reinterpret_cast<const float2*>(&s.fa.Sf[J][col]);
                const float2 db = *reinterpret_cast<const float2*>(&s.fa.Db[J][col]);
                const float2 emv = *reinterpret_cast<const float2*>(s.em + a);
                const float2 kpv = *reinterpret_cast<const float2*>(s.kp + a);
                const float dKbv[2] = {dKb2.x, dKb2.y}, sfx[2] = {sf.x, sf.y}, dbx[2] = {db.x, db.y},
                            emx[2] = {emv.x, emv.y}, kpx[2] = {kpv.x, kpv.y};
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int e = hh * 2 + e2;
                    const float ep = __fdividef(dbx[e2], emx[e2]);
                    adk[nt][e] += ep * acc[nt][e];
                    adg[nt][e] -= kpx[e2] * acc[nt][e];
                    adk[nt][e] += dKbv[e2] * (ep * sfx[e2]);   // (c) elementwise terms of Kbar
                    pk[nt][e] = dKbv[e2] * (kpx[e2] * sfx[e2]);
                }
            }
    }
    __syncthreads();   // all reads of qe, ke, kp, em, dB, dA done
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int row = rb * SUB + gid + hh * 8, col = chw + nt * 8 + tig * 2, a = pidx(row, col);
            *reinterpret_cast<float2*>(s.qe + a) = make_float2(adq[nt][hh * 2], adq[nt][hh * 2 + 1]);
            *reinterpret_cast<float2*>(s.ke + a) = make_float2(adk[nt][hh * 2], adk[nt][hh * 2 + 1]);
            *reinterpret_cast<float2*>(s.kp + a) = make_float2(adg[nt][hh * 2], adg[nt][hh * 2 + 1]);
            *reinterpret_cast<float2*>(s.em + a) = make_float2(pk[nt][hh * 2], pk[nt][hh * 2 + 1]);
        }
    __syncthreads();
    // dB and dAqk are no longer read: the next tile's rows stream in during the chains below
    if (cn.L > 0) stage_tile(nxt, cn);

    // thread (row group rg, channel cc) owns rows 16 rg .. 16 rg + 15 of channel cc in the dg scan and gate chain
    constexpr int RG = kPairThreads / CH;   // row groups (threads per channel)
    const int cc = tid & (CH - 1), rg = tid >> 6;
    const float dtc = dt_bias[h * D + cb + cc];
    // L2-norm chains: dx = (dx^ - x^ (x^ . dx^)) / sqrt(|x|^2 + eps); the row dot products
    // from both halves of the channels (rows as in the preparation)
    {
        uint2 xq[RB], xk[RB];
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            const int r = 16 * b + 2 * warp + hl;
            xq[b] = xk[b] = make_uint2(0u, 0u);
            if (r < L) {
                const size_t base = ((size_t)(t0 + r) * Hqk + h / G) * D + cb + c4;
                xq[b] = *reinterpret_cast<const uint2*>(q + base);
                xk[b] = *reinterpret_cast<const uint2*>(k + base);
            }
        }
        float pq[RB], pkd[RB];
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            const int r = 16 * b + 2 * warp + hl;
            const float iq = s.inq[r], ik = s.ink[r];
            const float4 gq = *reinterpret_cast<const float4*>(s.qe + pidx(r, c4));
            const float4 gk = *reinterpret_cast<const float4*>(s.ke + pidx(r, c4));
            float qv[4], kv[4];
            un4(xq[b], qv); un4(xk[b], kv);
            pq[b] = (qv[0] * iq) * gq.x + (qv[1] * iq) * gq.y + (qv[2] * iq) * gq.z + (qv[3] * iq) * gq.w;
            pkd[b] = (kv[0] * ik) * gk.x + (kv[1] * ik) * gk.y + (kv[2] * ik) * gk.z + (kv[3] * ik) * gk.w;
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
#pragma unroll
            for (int b = 0; b < RB; ++b) {
                pq[b] += __shfl_xor_sync(kAll, pq[b], o);
                pkd[b] += __shfl_xor_sync(kAll, pkd[b], o);
            }
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            const int r = 16 * b + 2 * warp + hl;
            if ((lane & 15) < 2) {
                float* x = &s.xd[half][lane & 15][r];
                const float v = (lane & 15) == 0 ? pq[b] : pkd[b];
                *x = v;
                st_async_peer(x, &s.mb_xd, peer, v);
            }
        }
        __syncthreads();
        wait_peer(&s.mb_xd);
#pragma unroll
        for (int b = 0; b < RB; ++b) {
            const int r = 16 * b + 2 * warp + hl;
            if (r < L) {
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    float xv[4];
                    un4(which == 0 ? xq[b] : xk[b], xv);
                    const float inv = which == 0 ? s.inq[r] : s.ink[r];
                    const float dot = s.xd[0][which][r] + s.xd[1][which][r];
                    const float4 g = *reinterpret_cast<const float4*>((which == 0 ? s.qe : s.ke) + pidx(r, c4));
                    const float gv[4] = {g.x, g.y, g.z, g.w};
                    float dx[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) dx[e] = (gv[e] - (xv[e] * inv) * dot) * inv;
                    if (!kGrouped) {
                        const size_t base = ((size_t)(t0 + r) * H + h) * D + cb + c4;
                        *reinterpret_cast<uint2*>((which == 0 ? dq : dk) + base) =
                            make_uint2((uint32_t)f2bf(dx[0]) | ((uint32_t)f2bf(dx[1]) << 16),
                                       (uint32_t)f2bf(dx[2]) | ((uint32_t)f2bf(dx[3]) << 16));
                    } else {   // this value head's share of dq, dk; summed per group afterwards
                        float* share = reinterpret_cast<float*>(ws + qk_share_offset(lay));
                        share += (((size_t)(t0 + r) * H + h) * 2 + which) * D + cb + c4;
                        *reinterpret_cast<float4*>(share) = make_float4(dx[0], dx[1], dx[2], dx[3]);
                    }
                }
            }
        }
    }
    // dg: sums over rows per key channel
    //   dg_t = sum_{i>=t} dG'_i + sum_{i<t} dKbar_i Kbar_i + dgam exp(G_L)
    // blocked over RG contiguous row segments of SEG rows, one per thread of the channel:
    // segment sums first, then each segment from its offsets, in registers; the gate chain
    // follows on the same rows
    float* part = reinterpret_cast<float*>(ws + lay.part) + tile * (D + 4);
    {
        constexpr int SEG = C / RG;
        float* segE = scr;             // [RG][64] sums of the dKbar Kbar terms
        float* segK = scr + RG * CH;   // [RG][64] sums of dG'
        const int r0 = rg * SEG;
        float pe[SEG], pg[SEG];
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
            const bool v = r0 + i < L;
            pe[i] = v ? s.em[pidx(r0 + i, cc)] : 0.0f;
            pg[i] = v ? s.kp[pidx(r0 + i, cc)] : 0.0f;
        }
        float se = 0.0f, sk = 0.0f;
#pragma unroll
        for (int i = 0; i < SEG; ++i) { se += pe[i]; sk += pg[i]; }
        segE[rg * CH + cc] = se;
        segK[rg * CH + cc] = sk;
        __syncthreads();
        // the chains have read dq^ and dk^: this CTA's channels of the raw gate rows of the
        // tile stream into the dq^ tile during the scan (rows past the chunk are not read)
        for (int seg = tid; seg < C * (CH / 8); seg += kPairThreads) {
            const int r = seg >> 3, c8 = (seg & 7) * 8;
            if (r < L) cp_async16(stgc + r * CH + c8, g_raw + ((size_t)(t0 + r) * H + h) * D + cb + c8);
        }
        cp_async_commit();
        float run = 0.0f, rev = reinterpret_cast<const float*>(bg + BgOff::DGAM)[cb + cc] * s.fa.gl[cc];
        for (int g2 = 0; g2 < rg; ++g2) run += segE[g2 * CH + cc];
        for (int g2 = RG - 1; g2 > rg; --g2) rev += segK[g2 * CH + cc];
#pragma unroll
        for (int i = 0; i < SEG; ++i) {   // exclusive prefix of the Kbar terms
            const float p = pe[i];
            pe[i] = run;
            run += p;
        }
#pragma unroll
        for (int i = SEG - 1; i >= 0; --i) {   // dg of row r0 + i
            rev += pg[i];
            pg[i] = rev + pe[i];
        }
        cp_async_wait_all();
        __syncthreads();
        // gate chain: du = dg lb sigmoid'(a (g_raw + dt_bias)), dg_raw = du a
        float ddt = 0.0f, dA = 0.0f;
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
            const int r = r0 + i;
            if (r < L) {
                const float x = bf2f(stgc[r * CH + cc]) + dtc;
                const float dgr = pg[i] * lb * dsigmoidf(a_h * x) * a_h;
                dg_raw[((size_t)(t0 + r) * H + h) * D + cb + cc] = f2bf(dgr);
                ddt += dgr;
                dA += dgr * x;
            }
        }
        // RG threads per channel (row segments); combined below in a fixed order
        scr[(2 * RG + rg) * CH + cc] = ddt;
        scr[(3 * RG + rg) * CH + cc] = dA;
    }
    __syncthreads();
    if (tid < CH) {
        float a = 0.0f, b = 0.0f;
#pragma unroll
        for (int g = 0; g < RG; ++g) { a += scr[(2 * RG + g) * CH + tid]; b += scr[(3 * RG + g) * CH + tid]; }
        part[cb + tid] = a;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) b += __shfl_xor_sync(kAll, b, o);
        if (lane == 0) s.red[warp] = b;
    }
    if (half == 0 && tid < L) {
        const float db = reinterpret_cast<const float*>(wy + WyOff::DBETA)[tid];
        dbeta_raw[(size_t)(t0 + tid) * H + h] = f2bf(db * dsigmoidf(bf2f(beta_raw[(size_t)(t0 + tid) * H + h])));
    }
    __syncthreads();
    if (tid == 0) part[D + half] = s.red[0] + s.red[1];
    if (cn.L <= 0) break;
    tile_i = nxt;
    ci = cn;
    alog = alog_next;
    braw = braw_next;
    par ^= 1u;
    }
    // neither CTA leaves while the other may still write into it (only after a timed-out wait
    // can a write be outstanding here)
    cluster_arrive();
    cluster_wait();
}


// The instantiation for the plain or the grouped head layout (template kernels are not
// visible outside this file).
BwdPairKernel bwd_pair_kernel(bool grouped) {
    return grouped ? kda_bwd_pair_kernel<true> : kda_bwd_pair_kernel<false>;
}

// Grouped value heads: dq, dk of query/key head g at a token = the sum of the shares of its
// value heads g G .. g G + G - 1 (fp32, in that order), rounded once to bf16. The shares
// are [tokens][H][2][128] (dq, dk); each thread takes 4 channels of one (token,
// query/key head) row, 8 rows per CTA.
__global__ void __launch_bounds__(256)
    kda_qk_group_reduce_kernel(uint16_t* __restrict__ dq, uint16_t* __restrict__ dk, uint8_t* __restrict__ ws,
                               int64_t tokens, Layout lay) {
    if (read_status(ws) != 0) return;
    const int G = (int)lay.G, H = (int)lay.H, Hqk = H / G;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= tokens * Hqk) return;
    const int64_t t = row / Hqk;
    const int g = (int)(row - t * Hqk), c4 = 4 * (threadIdx.x & 31);
    const float* share = reinterpret_cast<const float*>(ws + qk_share_offset(lay));
#pragma unroll
    for (int which = 0; which < 2; ++which) {
        const float* src = share + (((size_t)t * H + (size_t)g * G) * 2 + which) * D + c4;
        float4 a = *reinterpret_cast<const float4*>(src);
        for (int j = 1; j < G; ++j) {
            const float4 b = *reinterpret_cast<const float4*>(src + (size_t)j * 2 * D);
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        }
        uint16_t* dst = (which == 0 ? dq : dk) + ((size_t)t * Hqk + g) * D + c4;
        *reinterpret_cast<uint2*>(dst) = make_uint2((uint32_t)f2bf(a.x) | ((uint32_t)f2bf(a.y) << 16),
                                                    (uint32_t)f2bf(a.z) | ((uint32_t)f2bf(a.w) << 16));
    }
}

// Deterministic sum of the per-chunk parameter partials, per head. CTA (h, g) sums the
// chunks g, g + 8, g + 16, ... of head h in order (each chunk holds one ddt_bias partial per
// channel and two dA_log partials, one per channel half) into the scratch region; the last
// of a head's eight CTAs to finish (a counter per head) adds the eight sums in the order
// g = 0 .. 7 and resets the counter. Empty chunk records only follow the last real chunk.
__global__ void __launch_bounds__(128)
    kda_param_reduce_kernel(int H, float* __restrict__ dA_log, float* __restrict__ ddt_bias,
                            uint8_t* __restrict__ ws, Layout lay) {
    const int h = blockIdx.x, g = blockIdx.y, c = threadIdx.x;
    if (read_status(ws) != 0) return;
    const ChunkInfo* chunks = reinterpret_cast<const ChunkInfo*>(ws + lay.chunks);
    const float* part = reinterpret_cast<const float*>(ws + lay.part);
    float* sums = reinterpret_cast<float*>(ws + param_scratch_offset(lay));
    int* cnt = reinterpret_cast<int*>(sums + (size_t)H * kParamGroups * (D + 4));
    __shared__ int nreal;
    __shared__ int last;
    if (c == 0) {
        int lo = 0, hi = (int)lay.nc_max;   // first empty record (binary search)
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (chunks[mid].L > 0) lo = mid + 1;
            else hi = mid;
        }
        nreal = lo;
    }
    __syncthreads();
    const int n = nreal;
    float acc = 0.0f, accA = 0.0f;
    for (int ch = g; ch < n; ch += kParamGroups) {
        const float* p = part + ((size_t)ch * H + h) * (D + 4);
        acc += p[c];
        if (c == 0) accA += p[D] + p[D + 1];
    }
    float* mine = sums + ((size_t)h * kParamGroups + g) * (D + 4);
    mine[c] = acc;
    if (c == 0) mine[D] = accA;
    __threadfence();
    __syncthreads();
    if (c == 0) last = atomicAdd(cnt + h, 1) == kParamGroups - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    const volatile float* all = sums + (size_t)h * kParamGroups * (D + 4);
    float tot = 0.0f, totA = 0.0f;
#pragma unroll
    for (int u = 0; u < kParamGroups; ++u) {
        tot += all[u * (D + 4) + c];
        if (c == 0) totA += all[u * (D + 4) + D];
    }
    ddt_bias[h * D + c] = tot;
    if (c == 0) {
        dA_log[h] = totA;
        cnt[h] = 0;   // ready for the next backward on this workspace
    }
}

}  // namespace kda
