// Closed-form tree verify on tcgen05 tensor cores, forward-substitution solve,
// one 64-node block (T <= 64), bf16 q/k/v, fp32 S0, fp32 accumulation.
//
// Method: canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed
// form" (Bole's Theorem 1):
//     (I + G) U = R,  R = diag(beta) (V - diag(gamma) K S0^T),
//     O = diag(gamma) Q S0^T + C U,
// carried by the inverse W = (I + G)^-1 (ancestor sparsity) and M = C W:
//     U = W R,   O = diag(gamma) Q S0^T + M R.
//
// One CTA (256 threads) owns one (stream b, head h).  Its two warp groups
// work concurrently:
//   solve warps 0-3:  tree prep (each node walks its parent chain: path
//       bitmask, depth, cumulative log2 gate); the Gram block AC = [Q;K] K^T
//       on tcgen05; C and G rows with the decay 2^(l2_i - l2_j) on the
//       root-path entries, compacted to path positions; W and M rows by
//       right-looking substitution along each node's root path (rows are
//       independent: W (I + G) = I, M (I + G) = C); [M; W] to shared memory
//       as bf16 hi + lo (the B operand of the output product).
//   state warps 4-7:  S0 rows -> bf16 hi + lo in tensor memory (the A
//       operand); X^T = S0 [Q;K]^T on tcgen05 (value columns on the TMEM
//       lanes, nodes on the columns); R^T = beta (V - gamma X_K)^T as bf16
//       hi + lo into tensor memory.
// Then R^T [M; W]^T by three bf16 products (hi*hi + hi*lo + lo*hi, ~15
// mantissa bits each side), and each warp stores 32 value columns of
// o = gamma X_Q + M R (warps 0-3) or U = W R (warps 4-7) for every node.
// Decay ratios are only ever 2^(l2_i - l2_j) with j on i's root path, so they
// lie in (0, 1] and never overflow ("Hard constraints", log-space gates).
#include "common.cuh"

namespace canopy {

namespace tcf {

constexpr int DV = 128;
constexpr int TP = 64;    // nodes per block
constexpr int NT = 256;   // threads per CTA
constexpr int XS = 68;        // row stride (floats) of the work vectors and Gp: paths of up to 64 nodes
constexpr int XS_SHORT = 36;  // the same for paths of up to 33 nodes (depth <= 32)
constexpr uint32_t kTmemCols = 256;
// tensor-memory columns
constexpr uint32_t TA = 0;      // S0 as A: hi [0,64), lo [64,128); later R^T: hi [0,32), lo [32,64), and
                                // the output product's o part R^T M^T at [64,128)
constexpr uint32_t TD = 128;    // AC [128,192) first; then X^T [128,256): Q part [128,192), K part
                                // [192,256), the latter overwritten by the U part R^T W^T

struct Smem {
    static constexpr int QK = 0;                 // [Q;K] bf16, 2 atoms x 128 rows x 128 B; later [M;W] hi/lo
    static constexpr int BH = 0;                 // [M;W] bf16 hi: 128 rows x 128 B
    static constexpr int BL = 16384;             // [M;W] bf16 lo
    static constexpr int VT = 32768;             // V bf16: 2 tiles [64 nodes][64 cols], 128-byte swizzle
    static constexpr int V_TILE = 64 * 128;
    static constexpr int XV = VT + 2 * V_TILE;   // per-row work vectors fp32 [128][XS]
    static constexpr int GP = XV + 128 * XS * 4; // Gp fp32 [64][XS]: G rows by path position
    // trees of depth <= 32: work vectors and Gp with the short stride, clear
    // of the S0 staging area (so the solve runs while S0 is on its way)
    static constexpr int XV_SHORT = 65536;
    static constexpr int GP_SHORT = XV_SHORT + 128 * XS_SHORT * 4;
    static constexpr int PAR = GP + TP * XS * 4; // int[64] parent
    static constexpr int LEN = PAR + 256;        // int[64] path length
    static constexpr int L2 = LEN + 256;         // float[64] log2 gate, then cumulative
    static constexpr int GAM = L2 + 256;         // float[64] gamma
    static constexpr int BETA = GAM + 256;       // float[64]
    static constexpr int MASK = BETA + 256;      // u64[64] path(i), i included
    static constexpr int BAR = MASK + 512;       // u64[12]
    static constexpr int TMEMSLOT = BAR + 96;    // u32
    static constexpr int FLAG = TMEMSLOT + 4;    // int: a wait gave up
    static constexpr int NMAX = FLAG + 4;        // int: longest root path (nodes)

    static constexpr int BG = BAR + 128;         // float2[64] (beta, beta gamma)
    static constexpr int PLIST = BG + 512;       // u8[64][64] path(i) from the root down
    static constexpr int TOTAL = PLIST + TP * TP;
    // the S0 tile (fp32, 4 boxes of [128 rows][32 columns], 128-byte
    // swizzle) passes through a two-box staging area, one slot per box;
    // V and the long-stride tables reuse it once it has been converted
    static constexpr int S0S = 32768;
    static constexpr int S0_BOX = 128 * 128;
    static_assert(S0S + 2 * S0_BOX <= XV_SHORT && S0S % 1024 == 0, "S0 staging");
    static_assert(XV % 16 == 0 && GP % 16 == 0 && BAR % 256 == 0 && BG % 16 == 0 && GAM % 16 == 0, "align");
    static_assert(NMAX + 4 <= BG, "small arrays overlap");
    static_assert(GP_SHORT + TP * XS_SHORT * 4 <= PAR, "short tables overlap the small arrays");
};

enum { BAR_QK = 0, BAR_V, BAR_PREP, BAR_AC, BAR_ACC, BAR_X, BAR_Y, BAR_YU, BAR_S0, BAR_S0B, BAR_SFREE, NBAR };
static_assert(BAR_S0B == BAR_S0 + 1, "S0 slot barriers");
static_assert(NBAR <= 12, "barrier slots");

struct Params {
    const float* g;
    const float* beta;
    const int32_t* parent;
    const int32_t* lengths;  // per-stream node counts, or null (T everywhere)
    void* o;
    float* U;
    float* l;
    int32_t* depth;
    uint32_t* mask;
    int32_t* err;
    int B, T, H, W, o_bf16;
    int ratio;    // value heads per key head: value head h reads q and k of key head h / ratio
    float scale;  // factor on q: folded into gamma of the X_Q columns and into the M rows
    int inputs_ready;  // the inputs other than S0 may be read before the preceding kernel completes
    int state_ready;   // with inputs_ready: S0 too
};

// Two-part bf16 split with integer operations only (the conversion unit is
// a quarter-rate pipe, and these splits run for every S0, R and [M; W]
// element): hi = x rounded half-up to 8 significant bits, lo = x - hi
// (exact in fp32), and the lo kept as its top 16 bits (truncated), so
// |x - (hi + lo16)| < 2^-15 |x|.
__device__ inline uint32_t hi_bits(float x) { return (__float_as_uint(x) + 0x8000u) & 0xFFFF0000u; }
// bf16 pair from the top halves of two fp32 words: a -> low half, b -> high half.
__device__ inline uint32_t pack_top(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }
// Split x0, x1 into packed bf16 hi and lo pairs.
__device__ inline void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const uint32_t h0 = hi_bits(x0), h1 = hi_bits(x1);
    hi = pack_top(h0, h1);
    lo = pack_top(__float_as_uint(x0 - __uint_as_float(h0)), __float_as_uint(x1 - __uint_as_float(h1)));
}

__device__ inline void wait_or_flag(uint64_t* bar, int* sFlag) {
    if (!mbar_wait(bar, 0)) *sFlag = 1;
}

// One pass of R^T = beta (V - gamma X_K)^T over 32 nodes (hb = 0: nodes
// 0..31, hb = 1: 32..63) for value column c (this thread's TMEM lane): X_K
// from the accumulator columns, V from the shared tile, the result as bf16
// hi + lo into the A-operand columns.
__device__ __forceinline__ void r_pass(int hb, const uint8_t* sm, const float2* sBG, uint32_t lane_base, int c,
                                       int T) {
    const uint8_t* vt = sm + Smem::VT + (c >> 6) * Smem::V_TILE;
    const int cb = ((c & 63) >> 3), cw = (c & 7) << 1;
    uint32_t xk[32];
    tmem_ld16(lane_base + TD + 64 + hb * 32, *reinterpret_cast<uint32_t(*)[16]>(xk));
    tmem_ld16(lane_base + TD + 64 + hb * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(xk + 16));
    tmem_wait_ld();
    uint32_t wh[16], wl[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        float rv[2];
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
            const int i = hb * 32 + 2 * e + s2;
            const float vv = __bfloat162float(
                *reinterpret_cast<const __nv_bfloat16*>(vt + i * 128 + ((cb ^ (i & 7)) << 4) + cw));
            const float2 bg = sBG[i];
            // nodes past the stream's length are exactly zero (their rows may hold anything)
            rv[s2] = (i < T) ? bg.x * vv - bg.y * __uint_as_float(xk[2 * e + s2]) : 0.f;
        }
        split2(rv[0], rv[1], wh[e], wl[e]);
    }
    tmem_st16(lane_base + TA + hb * 16, wh);
    tmem_st16(lane_base + TA + 32 + hb * 16, wl);
}

__global__ void __launch_bounds__(NT, 2)
    verify_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmS,
                      Params p) {
    using L = Smem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* sPar = reinterpret_cast<int*>(sm + L::PAR);
    int* sLen = reinterpret_cast<int*>(sm + L::LEN);
    float* sL2 = reinterpret_cast<float*>(sm + L::L2);
    float* sGam = reinterpret_cast<float*>(sm + L::GAM);
    float* sBeta = reinterpret_cast<float*>(sm + L::BETA);
    uint64_t* sMask = reinterpret_cast<uint64_t*>(sm + L::MASK);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + L::TMEMSLOT);
    int* sFlag = reinterpret_cast<int*>(sm + L::FLAG);
    int* sNmax = reinterpret_cast<int*>(sm + L::NMAX);

    uint8_t* sPath = sm + L::PLIST;
    float2* sBG = reinterpret_cast<float2*>(sm + L::BG);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;                  // TMEM lane quadrant of this warp
    const bool solve = warp < 4;
    const int h = blockIdx.x, b = blockIdx.y;
    const int Ts = p.T, H = p.H;  // Ts: the stride of every [B][T] array
    int lbad = 0;
    const int T = stream_len(p.lengths, b, Ts, &lbad);  // this stream's nodes

    // Programmatic dependent launch: the next kernel may begin launching at
    // once.  With inputs_ready, until the preceding kernel has completed
    // (pdl_wait, by the thread that requests S0) only q, k, v, g, beta and
    // parent are read and nothing global is written; S0, the workspace and o
    // come after.  With state_ready as well, S0 is read early too, and only
    // the writes wait (each writing thread waits itself).  Otherwise
    // everything waits.
    if (!p.inputs_ready) pdl_wait();
    pdl_trigger();
    // Parents and gates first (threads 0..63), so that these small loads
    // enter the memory system ahead of the tile copies below.
    int par = -1;
    float ga = 1.f, gb = 0.f;
    if (tid < TP && tid < T) {
        par = p.parent[size_t(b) * Ts + tid];
        ga = p.g[(size_t(b) * Ts + tid) * H + h];
        gb = p.beta[(size_t(b) * Ts + tid) * H + h];
    }
    uint8_t* sQK = sm + L::QK;
    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *sFlag = 0;
        *sNmax = 0;
        // Q and K next: the solve path waits on them
        mbar_expect_tx(&bars[BAR_QK], 4 * 64 * 64 * 2);
        const int hk = (p.ratio == 1) ? h : h / p.ratio;
        tma_load_4d(sQK + 0, &tmQ, &bars[BAR_QK], 0, hk, 0, b);
        tma_load_4d(sQK + 16384, &tmQ, &bars[BAR_QK], 64, hk, 0, b);
        tma_load_4d(sQK + 8192, &tmK, &bars[BAR_QK], 0, hk, 0, b);
        tma_load_4d(sQK + 24576, &tmK, &bars[BAR_QK], 64, hk, 0, b);
    }
    if (warp == 0) {
        tmem_alloc(sTmem, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    // Validate; padded nodes: no path, beta 0, gamma 1.  Error bits are kept
    // and raised with the tree outputs, after the preceding kernel is done.
    int bad = (tid == 0) ? lbad : 0;
    if (tid < TP) {
        const int i = tid;
        if (i < T) {
            if (!((i == 0) ? (par == -1) : (par >= 0 && par < i))) {
                bad |= CANOPY_DEVERR_TREE;
                par = (i == 0) ? -1 : 0;
            }
            if (!gate_ok(ga, gb)) {
                bad |= CANOPY_DEVERR_GATE;
                ga = 1.f;
                gb = 0.f;
            }
        }
        sPar[i] = par;
        sL2[i] = log2f(ga);
        sBeta[i] = gb;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);


    if (solve) {
        // ---- tree prep: node i walks its (sanitised) parent chain ----------
        float myl2 = 0.f;
        if (tid < TP) {
            const int i = tid;
            uint64_t m = 0;
            int n = 0;
            if (i < T) {
                float s = 0.f;
                for (int j = i; j >= 0; j = sPar[j]) {
                    m |= 1ull << j;
                    s += sL2[j];
                    ++n;
                }
                myl2 = s;
            }
            sMask[i] = m;
            sLen[i] = n;
            atomicMax(sNmax, n);
        }
        group_sync(1, 128);
        if (tid < TP) {
            const int i = tid;
            sL2[i] = myl2;  // every walk has read the per-node gates by now
            const float gm = exp2f(myl2);
            sGam[i] = p.scale * gm;  // o = scale (gamma X_Q + M R): the X_Q columns' factor
            sBG[i] = make_float2(sBeta[i], sBeta[i] * gm);  // zero for padded nodes
            if (i < T) {
                int d = 0;
                for (uint64_t bits = sMask[i]; bits; bits &= bits - 1)
                    sPath[i * TP + d++] = uint8_t(__ffsll(static_cast<long long>(bits)) - 1);
            }
        }
        group_sync(1, 128);
        if (tid == 0) mbar_arrive(&bars[BAR_PREP]);  // gamma is ready for the state warps

        // ---- C and G rows from AC (lane r: Q row r, or K row r - 64) ----------
        // Trees of depth <= 32 keep their tables (short stride) clear of the
        // S0 staging area; deeper trees use the long stride over it and wait
        // until S0 has been converted.
        const bool shortp = *sNmax <= XS_SHORT - 3;
        const int xs = shortp ? XS_SHORT : XS;
        float* sX = reinterpret_cast<float*>(sm + (shortp ? L::XV_SHORT : L::XV));
        float* sGp = reinterpret_cast<float*>(sm + (shortp ? L::GP_SHORT : L::GP));
        const int r = tid;                     // 0..127: TMEM lane of this thread
        const bool qrow = r < TP;
        const int i = r & (TP - 1);
        float* xr = sX + r * xs;               // this row's work vector
        wait_or_flag(&bars[BAR_AC], sFlag);
        tc_fence_after();
        // The raw row goes to this thread's private array (local memory,
        // cached in L1): it is gathered by node index below, and shared
        // memory has no room for it next to the S0 staging.
        float raw[TP];
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
            uint32_t a[32];
            tmem_ld16(lane_base + TD + hc * 32, *reinterpret_cast<uint32_t(*)[16]>(a));
            tmem_ld16(lane_base + TD + hc * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(a + 16));
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) raw[hc * 32 + jj] = __uint_as_float(a[jj]);
        }
        tc_fence_before();
        group_sync(1, 128);
        if (tid == 0) mbar_arrive(&bars[BAR_ACC]);  // the AC columns may be overwritten
        if (!shortp) wait_or_flag(&bars[BAR_SFREE], sFlag);

        const int n = (i < T) ? sLen[i] : 0;
        const uint8_t* pl = sPath + i * TP;
        const float li = sL2[i];
        // C row (Q lanes) or G row (K lanes, strict ancestors, scaled by beta)
        // by path position, eight positions per batch (the raw row is in
        // local memory, and its loads should overlap).
        {
            const int cnt = qrow ? n : n - 1;
            float* dst = qrow ? xr : sGp + i * xs;
            const float sc = qrow ? 1.f : sBeta[i];
            for (int d0 = 0; d0 < cnt; d0 += 8) {
                int jj[8];
                float rv[8], lv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) jj[u] = pl[min(d0 + u, cnt - 1)];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    rv[u] = raw[jj[u]];
                    lv[u] = sL2[jj[u]];
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (d0 + u < cnt) dst[d0 + u] = sc * exp2f(li - lv[u]) * rv[u];
            }
            if (!qrow && n > 0) {
                // Gp row zero-padded by 4; the work vector becomes e_(n-1)
#pragma unroll
                for (int z = 0; z < 4; ++z) dst[n - 1 + z] = 0.f;
                for (int d = 0; d < n; ++d) xr[d] = (d == n - 1) ? 1.f : 0.f;
            }
        }
        group_sync(1, 128);

        // ---- W and M rows: right-looking substitution along path(i) ----------
        // x_d -= x_e Gp[pl[e]][d] for e = n-1 .. 1 and d < e, four pivots per
        // pass: the group of positions 4G..4G+3 is resolved in registers
        // (its pivots are final once every higher position has been applied),
        // then all four are applied to the groups below in one sweep.  Gp
        // rows are zero from their own position for four entries, so whole
        // groups are safe; pivots past the path count as zero.
        if (n > 1) {
            int G = (n - 1) >> 2;
            float4 xg = *reinterpret_cast<const float4*>(xr + 4 * G);
            for (;;) {
                const int base = 4 * G;
                int a[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) a[q] = pl[min(base + q, n - 1)];
                float xv[4] = {xg.x, xg.y, xg.z, xg.w};
#pragma unroll
                for (int q = 3; q >= 1; --q) {
                    const float4 gq = *reinterpret_cast<const float4*>(sGp + a[q] * xs + base);
                    const float pv = (base + q < n) ? xv[q] : 0.f;
                    if (q > 0) xv[0] -= pv * gq.x;
                    if (q > 1) xv[1] -= pv * gq.y;
                    if (q > 2) xv[2] -= pv * gq.z;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (base + q >= n) xv[q] = 0.f;
                *reinterpret_cast<float4*>(xr + base) = make_float4(xv[0], xv[1], xv[2], xv[3]);
                if (G == 0) break;
                const float* g0 = sGp + a[0] * xs;
                const float* g1 = sGp + a[1] * xs;
                const float* g2 = sGp + a[2] * xs;
                const float* g3 = sGp + a[3] * xs;
#pragma unroll 2
                for (int g = G - 1; g >= 0; --g) {
                    float4 x4 = *reinterpret_cast<const float4*>(xr + 4 * g);
                    const float4 h0 = *reinterpret_cast<const float4*>(g0 + 4 * g);
                    const float4 h1 = *reinterpret_cast<const float4*>(g1 + 4 * g);
                    const float4 h2 = *reinterpret_cast<const float4*>(g2 + 4 * g);
                    const float4 h3 = *reinterpret_cast<const float4*>(g3 + 4 * g);
                    x4.x -= xv[0] * h0.x + xv[1] * h1.x + xv[2] * h2.x + xv[3] * h3.x;
                    x4.y -= xv[0] * h0.y + xv[1] * h1.y + xv[2] * h2.y + xv[3] * h3.y;
                    x4.z -= xv[0] * h0.z + xv[1] * h1.z + xv[2] * h2.z + xv[3] * h3.z;
                    x4.w -= xv[0] * h0.w + xv[1] * h1.w + xv[2] * h2.w + xv[3] * h3.w;
                    if (g == G - 1)
                        xg = x4;  // the next pass's group stays in registers
                    else
                        *reinterpret_cast<float4*>(xr + 4 * g) = x4;
                }
                --G;
            }
        }

        // ---- [M; W] row r -> B operand (K-major bf16, 128-byte swizzle) ---------
        wait_or_flag(&bars[BAR_X], sFlag);  // the [Q;K] tile is no longer read
        {
            uint8_t* bh = sm + L::BH + r * 128;
            uint8_t* bl = sm + L::BL + r * 128;
            // zero the row chunk by chunk in swizzled order, so that the eight
            // rows of a quarter-warp write eight different bank groups
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                *reinterpret_cast<uint4*>(bh + ((c ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(bl + ((c ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
            }
            const float msc = qrow ? p.scale : 1.f;  // M rows carry the scale on q, W rows do not
            for (int d = 0; d < n; ++d) {
                const int j = pl[d];
                const float x = msc * xr[d];
                const uint32_t hb = hi_bits(x);
                const int off = ((((j >> 3) ^ (r & 7))) << 4) + ((j & 7) << 1);
                *reinterpret_cast<uint16_t*>(bh + off) = uint16_t(hb >> 16);
                *reinterpret_cast<uint16_t*>(bl + off) = uint16_t(__float_as_uint(x - __uint_as_float(hb)) >> 16);
            }
        }
        fence_proxy_async_smem();
        // tree outputs for the commit: l (natural log), depth, strict-ancestor
        // mask, once the preceding kernel has completed
        if (tid < TP) pdl_wait();
        if (bad) raise_err(p.err, bad);
        if (tid < TP && tid < T) {
            p.l[(size_t(b) * Ts + tid) * H + h] = sL2[tid] * 0.69314718055994531f;
            if (h == 0) {
                p.depth[size_t(b) * Ts + tid] = sLen[tid] - 1;
                const uint64_t strict = sMask[tid] & ~(1ull << tid);
                for (int w = 0; w < p.W; ++w)
                    p.mask[(size_t(b) * Ts + tid) * p.W + w] = uint32_t(strict >> (32 * w));
            }
        }

    } else {
        // ---- state warps: S0 rows -> bf16 hi/lo A operand in tensor memory ----
        // AC = [Q;K] K^T (M = 128, N = 64) as soon as Q and K have landed;
        // then V and S0 are requested (Q and K come first from HBM).
        const int c = quad * 32 + lane;  // value column of this thread in the R and store phases
        if (tid == 128) {
            if (mbar_wait(&bars[BAR_QK], 0)) {
                tc_fence_after();
                const uint32_t aQK = smem_u32(sQK);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t da = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                    const uint64_t db = sdesc_sw128(aQK + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32);
                    mma_bf16_ss(tmem + TD, da, db, idesc_bf16(128, 64), ks != 0);
                }
            } else {
                *sFlag = 1;
            }
            mma_commit(&bars[BAR_AC]);
            // S0 only once the preceding kernel of the stream has completed,
            // unless the caller says it does not write S0
            if (!p.state_ready) pdl_wait();
            for (int i = 0; i < 2; ++i) {
                mbar_expect_tx(&bars[BAR_S0 + i], L::S0_BOX);
                tma_load_4d(sm + L::S0S + i * L::S0_BOX, &tmS, &bars[BAR_S0 + i], 32 * i, 0, h, b);
            }
        }
        __syncwarp();
        // S0 row c (landed in shared memory by the copy engine) -> bf16 hi/lo
        // pairs in tensor-memory lane c; the 128-byte swizzle makes these
        // row-per-thread reads conflict-free.  The four boxes (32 keys each)
        // pass through two slots: box i uses slot i & 1 (barrier BAR_S0 +
        // (i & 1), phase i >> 1), and a slot is requested again as soon as
        // its box has been read.
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
            const int slot = i & 1;
            if (!mbar_wait(&bars[BAR_S0 + slot], uint32_t(i >> 1))) *sFlag = 1;
            const uint8_t* rowp = sm + L::S0S + slot * L::S0_BOX + c * 128;
            uint32_t wh[16], wl[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 f = *reinterpret_cast<const float4*>(rowp + ((j ^ (c & 7)) << 4));
                split2(f.x, f.y, wh[2 * j], wl[2 * j]);
                split2(f.z, f.w, wh[2 * j + 1], wl[2 * j + 1]);
            }
            tmem_st16(lane_base + TA + i * 16, wh);
            tmem_st16(lane_base + TA + 64 + i * 16, wl);
            tmem_wait_st();
            tc_fence_before();
            group_sync(2, 128);  // every thread has read (and stored) box i
            if (tid == 128) {
                if (i < 2) {
                    mbar_expect_tx(&bars[BAR_S0 + slot], L::S0_BOX);
                    tma_load_4d(sm + L::S0S + slot * L::S0_BOX, &tmS, &bars[BAR_S0 + slot], 32 * (i + 2), 0, h,
                                b);
                }
                if (i == 3) {
                    mbar_arrive(&bars[BAR_SFREE]);  // the staging area is free: V, then the solve tables
                    mbar_expect_tx(&bars[BAR_V], 2 * L::V_TILE);
                    tma_load_4d(sm + L::VT, &tmV, &bars[BAR_V], 0, h, 0, b);
                    tma_load_4d(sm + L::VT + L::V_TILE, &tmV, &bars[BAR_V], 64, h, 0, b);
                }
                if (i & 1) {
                    // X^T = S0 [Q;K]^T (M = 128 value rows, N = 128 nodes)
                    // over the 64 keys of boxes i - 1 and i (hi and lo
                    // parts); the first half goes while boxes 2 and 3 are
                    // on their way.  The AC columns must have been read out
                    // before X overwrites them.
                    const int hv = i >> 1;
                    if (hv == 0 && !mbar_wait(&bars[BAR_ACC], 0)) *sFlag = 1;
                    tc_fence_after();
                    const uint32_t aQK = smem_u32(sQK);
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const int ks = 4 * hv + k4;
                            const uint64_t db = sdesc_sw128(aQK + hv * 16384 + k4 * 32);
                            mma_bf16_ts(tmem + TD, tmem + TA + part * 64 + ks * 8, db, idesc_bf16(128, 128),
                                        (hv | part | k4) != 0);
                        }
                    if (hv == 1) mma_commit(&bars[BAR_X]);
                }
            }
        }
        __syncwarp();

        // ---- R^T = beta (V - gamma X_K)^T ---------------------------------------
        wait_or_flag(&bars[BAR_X], sFlag);
        wait_or_flag(&bars[BAR_V], sFlag);
        wait_or_flag(&bars[BAR_PREP], sFlag);
        tc_fence_after();
        {
            r_pass(0, sm, sBG, lane_base, c, T);
            r_pass(1, sm, sBG, lane_base, c, T);
            tmem_wait_st();
        }
        tc_fence_before();
    }
    __syncthreads();

    // ---- R^T [M; W]^T (bf16 x3): o part into the free S0 columns, U part
    // over X_K -------------------------------------------------------------------
    // o columns first, with their own commit: o (gamma X_Q added in the
    // epilogue) is stored while the U product runs.
    if (tid == 128) {
        tc_fence_after();
        const uint32_t bH = smem_u32(sm + L::BH), bL = smem_u32(sm + L::BL);
#pragma unroll 1
        for (int part = 0; part < 2; ++part) {        // 0: o (M rows), 1: U (W rows)
            const uint32_t d = tmem + (part ? TD + 64 : TA + 64);
            const uint32_t rowoff = part * 64 * 128;
#pragma unroll 1
            for (int pass = 0; pass < 3; ++pass) {    // hi*hi, hi*lo, lo*hi
                const uint32_t acol = TA + (pass == 2 ? 32 : 0);
                const uint32_t bb = (pass == 1 ? bL : bH) + rowoff;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_ts(d, tmem + acol + ks * 8, sdesc_sw128(bb + ks * 32), idesc_bf16(128, 64),
                                pass != 0 || ks != 0);
            }
            mma_commit(&bars[part ? BAR_YU : BAR_Y]);
        }
    }
    __syncwarp();
    wait_or_flag(&bars[solve ? BAR_Y : BAR_YU], sFlag);
    tc_fence_after();

    // ---- store: warps 0-3 o = gamma X_Q + R^T M^T, warps 4-7 U (lane = value
    // column), straight from the accumulator columns: per node row a warp
    // writes 32 consecutive columns (128 bytes of fp32, 64 of bf16); rows past
    // T are not written.  Writes wait until the preceding kernel has
    // completed. ---
    {
        const int c = quad * 32 + lane;
        const uint32_t col0 = solve ? TA + 64 : TD + 64;
        const size_t rstride = size_t(H) * DV;  // one node row of o or U
        const size_t base = (size_t(b) * Ts * H + h) * DV + c;
        pdl_wait();
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            uint32_t y[32];
            tmem_ld16(lane_base + col0 + half * 32, *reinterpret_cast<uint32_t(*)[16]>(y));
            tmem_ld16(lane_base + col0 + half * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(y + 16));
            const int e0 = half * 32;
            if (solve) {
                uint32_t xq[32];
                tmem_ld16(lane_base + TD + half * 32, *reinterpret_cast<uint32_t(*)[16]>(xq));
                tmem_ld16(lane_base + TD + half * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(xq + 16));
                tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    // sGam carries the scale on q
                    const float4 gm = *reinterpret_cast<const float4*>(sGam + e0 + 4 * e4);
                    y[4 * e4] = __float_as_uint(fmaf(gm.x, __uint_as_float(xq[4 * e4]), __uint_as_float(y[4 * e4])));
                    y[4 * e4 + 1] =
                        __float_as_uint(fmaf(gm.y, __uint_as_float(xq[4 * e4 + 1]), __uint_as_float(y[4 * e4 + 1])));
                    y[4 * e4 + 2] =
                        __float_as_uint(fmaf(gm.z, __uint_as_float(xq[4 * e4 + 2]), __uint_as_float(y[4 * e4 + 2])));
                    y[4 * e4 + 3] =
                        __float_as_uint(fmaf(gm.w, __uint_as_float(xq[4 * e4 + 3]), __uint_as_float(y[4 * e4 + 3])));
                }
            } else {
                tmem_wait_ld();
            }
            if (solve && p.o_bf16) {
                __nv_bfloat16* op = static_cast<__nv_bfloat16*>(p.o) + base;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e0 + e < T) op[(e0 + e) * rstride] = __float2bfloat16_rn(__uint_as_float(y[e]));
            } else {
                float* op = solve ? static_cast<float*>(p.o) + base : p.U + base;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e0 + e < T) op[(e0 + e) * rstride] = __uint_as_float(y[e]);
            }
        }
    }
    if (tid == 128 && *sFlag) {
        // a wait gave up: let the copies in flight land before leaving
        raise_err(p.err, CANOPY_DEVERR_TIMEOUT);
        // (thread 128 issued every S0 and V copy; each wait is bounded)
        mbar_wait(&bars[BAR_QK], 0);
        for (int i = 0; i < 4; ++i) mbar_wait(&bars[BAR_S0 + (i & 1)], uint32_t(i >> 1));
        mbar_wait(&bars[BAR_V], 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace tcf

// ---------------------------------------------------------------------------
// Host side.

bool make_bf16_row_map(CUtensorMap* m, const void* base, int B, int T, int H);
bool make_state_map(CUtensorMap* m, const float* base, int B, int H);

cudaError_t launch_verify_tc_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const float* S0, const int32_t* parent, const int32_t* lengths, int T, int B, int H,
                                 int HK, void* o, int o_bf16, float scale, const Ws& ws, int inputs_ready,
                                 int state_ready, cudaStream_t st) {
    CUtensorMap mq, mk, mv, ms;
    if (!make_bf16_row_map(&mq, q, B, T, HK) || !make_bf16_row_map(&mk, k, B, T, HK) ||
        !make_bf16_row_map(&mv, v, B, T, H) || !make_state_map(&ms, S0, B, H))
        return cudaErrorInvalidValue;
    tcf::Params prm;
    prm.g = g;
    prm.beta = beta;
    prm.parent = parent;
    prm.lengths = lengths;
    prm.o = o;
    prm.U = ws.U;
    prm.l = ws.l;
    prm.depth = ws.depth;
    prm.mask = ws.mask;
    prm.err = ws.err;
    prm.B = B;
    prm.T = T;
    prm.H = H;
    prm.W = ws.W;
    prm.o_bf16 = o_bf16;
    prm.ratio = H / HK;
    prm.scale = scale;
    prm.inputs_ready = inputs_ready;
    prm.state_ready = inputs_ready && state_ready;
    const int smem = tcf::Smem::TOTAL + 1024;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tcf::verify_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    return launch_pdl(tcf::verify_fwd_kernel, dim3(H, B), dim3(tcf::NT), smem, st, mq, mk, mv, ms, prm);
}

}  // namespace canopy
