// Commit kernel: rebuild only the accepted node's state.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form"
// (last line) and "What the commit kernel stores", in the (dv, dk)
// orientation:  S_new = gamma_a S0 + sum_{j in path(a)} exp(l_a - l_j) u_j k_j^T,
// all in fp32, from the U and l the verify call left in the workspace and
// that call's k and parent.
//
// Memory bound: every element of S0 is read once and S_new written once.
// One CTA (256 threads) rebuilds TPC 32-row tiles of a (stream, value head)
// state (the whole state at dv = 128), so the path walk and the path's k rows
// are fetched once per state.  At its start the CTA requests all its S0 tiles
// by bulk copy (all in flight at once).  The path's k rows and weighted u rows
// are staged in shared memory 32 nodes at a time, and the rank-n update of
// every tile is accumulated in registers, node by node, while the S0 tiles
// are still landing; each tile then adds gamma_a S0 and is stored as soon as
// it has landed.  The update uses packed two-lane fp32 FMAs (the same
// rounding as two scalar FMAs, half the instructions).  (Measured on GB300,
// commits back to back at B = 16, T = 64: 7.60 us with the update run tile
// by tile after each tile had landed, 7.13 with the parents requested ahead
// of S0, 6.74 with the update hoisted, 6.59 with packed FMAs.)
#include "common.cuh"

namespace canopy {

namespace cm {

constexpr int NT = 256;    // threads per CTA
constexpr int ROWS = 32;   // value rows per tile (one bulk copy)
constexpr int CH = 32;     // path nodes staged per pass
constexpr int TPC = 4;    // 32-row tiles per CTA (the whole state at dv = 128)

__device__ inline float4 k4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ inline float4 k4(const __nv_bfloat16* p) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
}

template <typename InT, int DK, int DV>
struct CommitSmem {
    static constexpr int NTILE = (DV / ROWS < TPC) ? DV / ROWS : TPC;
    static constexpr uint32_t TILE = ROWS * DK * 4;
    float s[NTILE * ROWS * DK];    // S0, then S_new, tile by tile
    InT k[CH][DK];                 // k rows of the current path chunk
    float wu[CH][DV];              // exp(l_a - l_j) u_j for the chunk's nodes, every value row
    int par[kMaxT];                // the stream's parents
    int path[kMaxT];               // path(a), a first
    uint64_t bar[TPC];
    int n, bad;
};

// Stage path nodes c0 .. c0 + cn - 1: their k rows, and (after the verify has
// completed) their weighted u rows.  Each thread issues all its loads before
// it stores any of them, so a chunk costs one memory round trip.
template <typename InT, int DK, int DV>
__device__ __forceinline__ void stage_k(CommitSmem<InT, DK, DV>& S, const InT* __restrict__ k, int b, int T, int HK,
                                        int hk, int c0, int cn) {
    constexpr int KV = 16 / sizeof(InT);  // k elements per 16-byte load
    constexpr int PER = DK / KV;          // 16-byte loads per k row
    constexpr int IT = (CH * PER + NT - 1) / NT;
    uint4 buf[IT];
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int e = threadIdx.x + i * NT;
        if (e < cn * PER) {
            const int r = e / PER, c = (e % PER) * KV, j = S.path[c0 + r];
            buf[i] = *reinterpret_cast<const uint4*>(k + ((size_t(b) * T + j) * HK + hk) * DK + c);
        }
    }
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int e = threadIdx.x + i * NT;
        if (e < cn * PER) *reinterpret_cast<uint4*>(&S.k[e / PER][(e % PER) * KV]) = buf[i];
    }
}
// la = l of the accepted node; with cn > 0 it is read here, in the same round
// trip as the chunk's l and u entries (path[0] is the accepted node).
template <typename InT, int DK, int DV>
__device__ __forceinline__ void stage_wu(CommitSmem<InT, DK, DV>& S, const Ws& ws, int b, int T, int H, int h,
                                         float& la, bool read_la, int c0, int cn) {
    constexpr int PER = DV / 4;
    constexpr int IT = (CH * PER + NT - 1) / NT;
    if (read_la) la = ws.l[(size_t(b) * T + S.path[0]) * H + h];
    float lj[IT];
    float4 u[IT];
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int e = threadIdx.x + i * NT;
        if (e < cn * PER) {
            const int r = e / PER, c = (e % PER) * 4;
            const size_t nh = (size_t(b) * T + S.path[c0 + r]) * H + h;
            lj[i] = ws.l[nh];
            u[i] = *reinterpret_cast<const float4*>(ws.U + nh * DV + c);
        }
    }
#pragma unroll
    for (int i = 0; i < IT; ++i) {
        const int e = threadIdx.x + i * NT;
        if (e < cn * PER) {
            const float w = expf(la - lj[i]);
            *reinterpret_cast<float4*>(&S.wu[e / PER][(e % PER) * 4]) =
                make_float4(w * u[i].x, w * u[i].y, w * u[i].z, w * u[i].w);
        }
    }
}

template <typename InT, int DK, int DV>
__global__ void __launch_bounds__(NT) commit_kernel(const int32_t* __restrict__ accepted,
                                                    const int32_t* __restrict__ parent,
                                                    const int32_t* __restrict__ lengths, const float* S0,
                                                    float* S_new, const InT* __restrict__ k, int T, int H, int HK,
                                                    Ws ws, int state_ready) {
    using Sm = CommitSmem<InT, DK, DV>;
    constexpr int NTILE = Sm::NTILE;
    constexpr int C4 = DK / 4;             // float4 per state row
    constexpr int RPT = ROWS * C4 / NT;    // rows of a tile per thread
    static_assert(NTILE <= TPC && NT % C4 == 0 && (ROWS * C4) % NT == 0 && RPT >= 1, "tile shape");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Sm& S = *reinterpret_cast<Sm*>(smem_raw);
    const int h = blockIdx.y, b = blockIdx.z, t = threadIdx.x;
    const int hk = h / (H / HK);  // the key head this value head reads
    // this thread: float4 column c4 of rows r0 .. r0 + RPT - 1 of every tile
    const int c4 = t % C4, r0 = (t / C4) * RPT;
    const int vbase = blockIdx.x * NTILE * ROWS;  // first value row of this CTA
    const size_t sbase = ((size_t(b) * H + h) * DV + vbase) * DK;

    // Programmatic dependent launch: with state_ready, the S0 tiles, the
    // accepted node, the parents and the path's k rows are read while the
    // preceding kernel finishes; the workspace and S_new only after it has
    // completed.
    if (!state_ready) pdl_wait();
    pdl_trigger();
    // Warp 0 requests the stream's parents, its length and the accepted node
    // before the S0 copies are issued, so that these few bytes (which the
    // path walk, and through it every later read, waits on) are not queued
    // behind the 64 KB of S0 per CTA.
    constexpr int PPL = kMaxT / 32;  // parents per lane
    int pj[PPL];
    int a = -1, len = T;
    if (t < 32) {
#pragma unroll
        for (int i = 0; i < PPL; ++i) {
            const int j = t + 32 * i;
            pj[i] = (j < T) ? parent[size_t(b) * T + j] : 0;
        }
        a = accepted[b];
        if (lengths) len = lengths[b];
    }
    if (t == 0) {
        for (int i = 0; i < NTILE; ++i) mbar_init(&S.bar[i], 1);
        fence_mbar_init();
        for (int i = 0; i < NTILE; ++i) {
            mbar_expect_tx(&S.bar[i], Sm::TILE);
            bulk_load(S.s + i * ROWS * DK, S0 + sbase + size_t(i) * ROWS * DK, Sm::TILE, &S.bar[i]);
        }
    }
    if (t < 32) {
        // the stream's nodes: lengths[b] of the T-strided arrays (all T without lengths)
        int lbad = 0;
        if (len < 0 || len > T) {
            lbad = CANOPY_DEVERR_LENGTH;
            len = len < 0 ? 0 : T;
        }
#pragma unroll
        for (int i = 0; i < PPL; ++i)
            if (t + 32 * i < len) S.par[t + 32 * i] = pj[i];
        __syncwarp();
        if (t == 0) {
            int bad = (a < -1 || a >= len) ? CANOPY_DEVERR_ACCEPTED : 0;
            if (bad) a = -1;
            bad |= lbad;
            // path(a) from a up to the root, parents sanitised as the verify
            // sanitises them (node 0 is the root; a parent outside [0, j)
            // reads as 0), so the walk ends within a + 1 steps
            int n = 0;
            for (int j = a; j >= 0;) {
                S.path[n++] = j;
                const int p = S.par[j];
                j = (j == 0) ? -1 : ((p >= 0 && p < j) ? p : 0);
            }
            S.n = n;
            S.bad = bad;
        }
    }
    __syncthreads();
    const int n = S.n;
    const int nch = (n + CH - 1) / CH;
    stage_k(S, k, b, T, HK, hk, 0, min(CH, n));
    if (state_ready) pdl_wait();
    if (S.bad && t == 0 && h == 0 && blockIdx.x == 0) raise_err(ws.err, S.bad);
    float la = 0.f;
    stage_wu(S, ws, b, T, H, h, la, n > 0, 0, min(CH, n));
    const float gamma_a = (n > 0) ? expf(la) : 1.f;
    __syncthreads();

    // The path's rank-n update first, for every tile of the state at once
    // (each node's k chunk is read once for the NTILE tiles, and the update
    // runs while the S0 tiles are still landing); then each tile, as it
    // lands, adds gamma_a S0 and is stored.
    float4 acc[NTILE][RPT];
#pragma unroll
    for (int tile = 0; tile < NTILE; ++tile)
#pragma unroll
        for (int u = 0; u < RPT; ++u) acc[tile][u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
        const int cn = min(CH, n - ch * CH);
        if (ch > 0) {
            // deep paths: the next chunk's k and u rows
            __syncthreads();
            stage_k(S, k, b, T, HK, hk, ch * CH, cn);
            stage_wu(S, ws, b, T, H, h, la, false, ch * CH, cn);
            __syncthreads();
        }
        for (int r = 0; r < cn; ++r) {
            const float4 kk = k4(&S.k[r][c4 * 4]);
#pragma unroll
            for (int tile = 0; tile < NTILE; ++tile) {
                float wv[RPT];
                if constexpr (RPT == 4) {
                    const float4 w4 = *reinterpret_cast<const float4*>(&S.wu[r][vbase + tile * ROWS + r0]);
                    wv[0] = w4.x;
                    wv[1] = w4.y;
                    wv[2] = w4.z;
                    wv[3] = w4.w;
                } else {
#pragma unroll
                    for (int u = 0; u < RPT; ++u) wv[u] = S.wu[r][vbase + tile * ROWS + r0 + u];
                }
#pragma unroll
                for (int u = 0; u < RPT; ++u) {
                    const float2 w2 = make_float2(wv[u], wv[u]);
                    float2 lo = __ffma2_rn(w2, make_float2(kk.x, kk.y), make_float2(acc[tile][u].x, acc[tile][u].y));
                    float2 hi = __ffma2_rn(w2, make_float2(kk.z, kk.w), make_float2(acc[tile][u].z, acc[tile][u].w));
                    acc[tile][u] = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
            }
        }
    }
    bool timeout = false;
#pragma unroll
    for (int tile = 0; tile < NTILE; ++tile) {
        const int v0 = tile * ROWS;  // relative to vbase
        if (!mbar_wait(&S.bar[tile], 0)) timeout = true;
        const float* st = S.s + tile * ROWS * DK;
#pragma unroll
        for (int u = 0; u < RPT; ++u) {
            const float4 s = *reinterpret_cast<const float4*>(st + ((r0 + u) * C4 + c4) * 4);
            float4 o = acc[tile][u];
            o.x = fmaf(gamma_a, s.x, o.x);
            o.y = fmaf(gamma_a, s.y, o.y);
            o.z = fmaf(gamma_a, s.z, o.z);
            o.w = fmaf(gamma_a, s.w, o.w);
            *reinterpret_cast<float4*>(S_new + sbase + size_t((v0 + r0 + u) * C4 + c4) * 4) = o;
        }
    }
    if (timeout && t == 0) raise_err(ws.err, CANOPY_DEVERR_TIMEOUT);
}

}  // namespace cm

template <typename InT, int D>
static cudaError_t launch_commit_typed(const int32_t* accepted, const int32_t* parent, const int32_t* lengths,
                                       const float* S0, float* S_new, const void* k, int T, int B, int H, int HK,
                                       const Ws& ws, int state_ready, cudaStream_t st) {
    const size_t smem = sizeof(cm::CommitSmem<InT, D, D>);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(cm::commit_kernel<InT, D, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int nt = (D / cm::ROWS < cm::TPC) ? D / cm::ROWS : cm::TPC;
    return launch_pdl(cm::commit_kernel<InT, D, D>, dim3(D / cm::ROWS / nt, H, B), dim3(cm::NT), smem, st, accepted,
                      parent, lengths, S0, S_new, static_cast<const InT*>(k), T, H, HK, ws, state_ready);
}

cudaError_t launch_commit(const int32_t* accepted, const int32_t* parent, const int32_t* lengths, const float* S0,
                          float* S_new, const void* k, int in_bf16, int T, int B, int H, int HK, int d, const Ws& ws,
                          int state_ready, cudaStream_t st) {
    using bf = __nv_bfloat16;
#define CANOPY_COMMIT(IT, D) \
    return launch_commit_typed<IT, D>(accepted, parent, lengths, S0, S_new, k, T, B, H, HK, ws, state_ready, st)
    if (d == 128) {
        if (in_bf16) CANOPY_COMMIT(bf, 128);
        CANOPY_COMMIT(float, 128);
    }
    if (in_bf16) CANOPY_COMMIT(bf, 32);
    CANOPY_COMMIT(float, 32);
#undef CANOPY_COMMIT
}

}  // namespace canopy
