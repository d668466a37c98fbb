// Closed-form tree verify on tcgen05 tensor cores for trees of 65 to 256
// nodes: bf16 q/k/v, fp32 S0, dk = dv = 128, forward-substitution solve, one
// launch, one CTA per (stream b, value head h).
//
// Method: canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed
// form" (Bole's Theorem 1), blocked as its "Design decisions" lays out: the
// 64-node diagonal blocks are solved in order and the off-diagonal updates
// are tensor-core products.  With value columns on the tensor-memory lanes
// (the (dv, dk) orientation), for block r (nodes 64 r .. 64 r + 63):
//     D  = S0 [Q_r; K_r]^T                                  (X_Q | X_K)
//     D <- (scale gamma X_Q | beta (V_r - gamma X_K))        R_r in the K half
//     D += U_s^T [scale C_rs; -G_rs]^T       for s < r       cross-block terms
//     R'_r = K half of D,  U_r = W_rr R'_r,  O_r = Q half of D + scale M_rr R'_r
// where W_rr = (I + G_rr)^-1 and M_rr = C_rr W_rr.  Their rows follow by
// substitution along each node's in-block root path (W (I + G) = I,
// M (I + G) = C: rows are independent, and the in-block path of an ancestor
// is a prefix of the node's own), exactly as in the single-block kernel.
//
// Tensor memory (512 columns): S0 as bf16 hi + lo (the A operand of every X
// product, converted once); the accumulator D; one Gram tile [Q_r; K_r] K_s^T
// at a time, whose columns later hold R'^T as bf16 hi + lo; and U_s^T as bf16
// hi + lo for the blocks later blocks read.  The Gram tiles, C, G, W and M
// never leave the chip: every product ([Q;K] K^T, S0 [Q;K]^T, the cross
// terms and R' [M; W]^T) runs on tcgen05 with fp32 accumulation, split bf16
// operands (hi + lo, three products) wherever an operand is not exact bf16.
//
// Warp roles, each role running its own loop over the blocks:
//   warps 0-3 (solve; one thread per row of [Q_r; K_r], i.e. per TMEM lane of
//       the Gram tile): read the Gram tiles, build the W and M rows of the
//       diagonal block and the [scale C_rs; -G_rs] rows of the cross terms
//       (only the entries on root paths are computed);
//   warps 4-7 (state; one thread per value column): convert S0, transform D,
//       form R', and store o and U through shared memory by bulk tensor
//       stores; thread 128 issues the X and output products and the Q_r/K_r,
//       V_r and S0 copies;
//   warp 8 (issuer): issues the Gram and cross-term products and the K_s
//       copies, so that no compute warp waits on a copy or a product it does
//       not consume.  Tile s + 1's Gram product runs while tile s's rows are
//       built, and two [C; -G] buffers let a build overlap the previous
//       cross-term product.  Every barrier a role waits on in sequence can
//       only complete its next phase after that role has acted on the one it
//       waited for (the two buffers have a "built" and a "consumed" barrier
//       each), so no phase is ever skipped.
// Every mbarrier wait is bounded: a timeout sets CANOPY_DEVERR_TIMEOUT and the
// later waits are skipped; before leaving, copies and products in flight are
// awaited (bounded) and tensor memory is freed.
#include "common.cuh"

namespace canopy {

namespace tcb {

constexpr int DV = 128;
constexpr int TP = 64;               // nodes per block
constexpr int NT = 288;              // threads per CTA: solve, state and issuer warps
constexpr int ISSUER = 256;          // first thread of the issuer warp
constexpr int MAXB = kMaxT / TP;     // blocks per tree at most
constexpr int XS = 68;               // row stride (floats) of the substitution tables
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TA = 0;           // S0^T operand: hi [0, 64), lo [64, 128)
constexpr uint32_t TD = 128;         // D: Q half [128, 192), K half [192, 256)
constexpr uint32_t TG = 256;         // Gram tile [256, 320); then R'^T hi [256, 288), lo [288, 320)
constexpr uint32_t TU = 320;         // U_s^T (s < MAXB - 1): hi [TU + 64 s, +32), lo [+32, +64)
static_assert(TU + 64 * (MAXB - 1) == kTmemCols, "tensor memory plan");

struct Smem {
    static constexpr int QK = 0;                     // [Q_r; K_r] bf16: 2 key atoms x 128 rows x 128 B
    static constexpr int KS = 32768;                 // two K_s slots: 2 key atoms x 64 rows x 128 B each
    static constexpr int KS_TILE = 16384;
    static constexpr int MWH = KS + 2 * KS_TILE;     // [scale M_rr; W_rr] bf16 hi: 128 rows x 128 B
    static constexpr int MWL = MWH + 16384;          // lo
    static constexpr int VT = MWL + 16384;           // V_r bf16: 2 tiles [64 nodes][64 columns]
    static constexpr int V_TILE = 8192;
    static constexpr int RX = VT + 2 * V_TILE;       // used in turn by the S0 staging, the diagonal
    static constexpr int S0_BOX = 16384;             //   block's tables and the two [C; -G] buffers
    static constexpr int XV = RX;                    // fp32 [128][XS] work vectors
    static constexpr int GP = XV + 128 * XS * 4;     // fp32 [64][XS] G rows by path position
    static constexpr int CG = RX;                    // [C; -G] buffer b: hi at CG + b CG_BUF, lo 16 KB on
    static constexpr int CG_BUF = 32768;
    static constexpr int RX_END = RX + 2 * CG_BUF;
    static constexpr int ST = RX_END;                // two store staging tiles [32 nodes][128 columns]
    static constexpr int ST_BUF = 16384;
    static constexpr int LEN = ST + 2 * ST_BUF;      // int[256] |path(i)|
    static constexpr int L2 = LEN + 1024;            // float[256] cumulative log2 gate
    static constexpr int GAM = L2 + 1024;            // float[256] gamma = 2^l2
    static constexpr int BETA = GAM + 1024;          // float[256]
    static constexpr int MASK = BETA + 1024;         // u64[256][4] path(i), i included
    static constexpr int PLIST = MASK + 8192;        // u8[64][64] in-block paths of the current block
    static constexpr int LSUM = PLIST;               // double[256] log2 gate sums (tree prep only)
    static constexpr int PAR = PLIST + 2048;         // int[256] parents, then jump pointers (tree prep only)
    static constexpr int NIN = PLIST + TP * TP;      // int[64] in-block path lengths
    static constexpr int BAR = NIN + 256;            // u64[32]
    static constexpr int TMEMSLOT = BAR + 256;
    static constexpr int FLAG = TMEMSLOT + 4;
    static constexpr int TOTAL = FLAG + 4;
    static_assert(KS % 1024 == 0 && MWH % 1024 == 0 && VT % 1024 == 0 && RX % 1024 == 0 && ST % 1024 == 0,
                  "tile alignment");
    static_assert(2 * S0_BOX <= RX_END - RX && GP + TP * XS * 4 <= RX_END, "region X");
    static_assert(PAR + 1024 <= NIN, "tree-prep arrays inside the path lists");
    static_assert(MASK % 8 == 0 && BAR % 8 == 0, "alignment");
    static_assert(TOTAL + 1024 <= 227 * 1024, "shared memory");
};

enum {
    BAR_QK = 0, BAR_V, BAR_S0, BAR_S0B, BAR_SFREE, BAR_KS0, BAR_KS1, BAR_G, BAR_X, BAR_XT, BAR_MW, BAR_TGF,
    BAR_CR0, BAR_CR1, BAR_W, BAR_DREAD, BAR_TREAD, BAR_CGB0, BAR_CGB1, BAR_PREP, NBAR
};
static_assert(NBAR <= 32 && BAR_S0B == BAR_S0 + 1 && BAR_KS1 == BAR_KS0 + 1 && BAR_CR1 == BAR_CR0 + 1 &&
                  BAR_CGB1 == BAR_CGB0 + 1,
              "barriers");

struct Params {
    const float* g;
    const float* beta;
    const int32_t* parent;
    const int32_t* lengths;  // per-stream node counts, or null (T everywhere)
    void* o;                 // written directly (not by bulk store) where a
    float* U;                //   stream ends inside a 32-node tile
    float* l;
    int32_t* depth;
    uint32_t* mask;
    int32_t* err;
    int B, T, H, W, o_bf16;
    int ratio;    // value heads per key head
    float scale;  // factor on q: on the Q half of D, and on the C and M rows
};

// Two-part bf16 split with integer operations only: hi = x rounded half-up to
// 8 significant bits, lo = the top 16 bits of x - hi (exact in fp32).
__device__ inline uint32_t hi_bits(float x) { return (__float_as_uint(x) + 0x8000u) & 0xFFFF0000u; }
__device__ inline uint32_t pack_top(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }
__device__ inline void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const uint32_t h0 = hi_bits(x0), h1 = hi_bits(x1);
    hi = pack_top(h0, h1);
    lo = pack_top(__float_as_uint(x0 - __uint_as_float(h0)), __float_as_uint(x1 - __uint_as_float(h1)));
}

// Bounded wait; once any wait of the CTA has given up, the later ones are
// skipped (the outputs are then undefined and the error word says so), so
// the CTA runs to its end quickly.
__device__ inline void wait_or_flag(uint64_t* bar, uint32_t parity, volatile int* sFlag) {
    if (*sFlag) return;
    if (!mbar_wait(bar, parity)) *sFlag = 1;
}

// Row rho's 64 Gram entries (lane rho of the tile) into raw[] (indexed by
// node below, so it lives in local memory, cached in L1).
__device__ __forceinline__ void read_gram_row(uint32_t lane_base, float (&raw)[TP]) {
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
        uint32_t a[32];
        tmem_ld16(lane_base + TG + hc * 32, *reinterpret_cast<uint32_t(*)[16]>(a));
        tmem_ld16(lane_base + TG + hc * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(a + 16));
        tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) raw[hc * 32 + jj] = __uint_as_float(a[jj]);
    }
}

// Issue [Q_r; K_r] B^T (M = 128, N = 64, K = 128) into the Gram columns; b_lo
// is the B tile's first key atom and b_atom the distance to its second.
__device__ __forceinline__ void issue_gram(uint32_t tmem, uint32_t aQK, uint32_t b_lo, uint32_t b_atom) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint64_t da = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
        const uint64_t db = sdesc_sw128(b_lo + (ks >> 2) * b_atom + (ks & 3) * 32);
        mma_bf16_ss(tmem + TG, da, db, idesc_bf16(128, 64), ks != 0);
    }
}

// Path bitmasks and root-path log2 gate sums by pointer jumping (as in
// jump_paths), run by the 128 solve threads alone, two nodes each, with
// their named barrier; ceil(log2 T) rounds cover every root path.
__device__ void jump_paths_solve(int T, int* sPtr, int* sLen, double* sS, uint64_t* sM) {
    const int t = threadIdx.x;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int i = t + 128 * u;
        if (i < T) {
#pragma unroll
            for (int w = 0; w < 4; ++w) sM[i * 4 + w] = (w == (i >> 6)) ? (1ull << (i & 63)) : 0ull;
            sLen[i] = 1;
        }
    }
    group_sync(1, 128);
    int rounds = 0;
    while ((1 << rounds) < T) ++rounds;
    for (int round = 0; round < rounds; ++round) {
        JumpState<4, double> st[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = t + 128 * u;
            if (i >= T) continue;
            const int pp = sPtr[i];
#pragma unroll
            for (int w = 0; w < 4; ++w) st[u].m[w] = sM[i * 4 + w];
            st[u].s = sS[i];
            st[u].len = sLen[i];
            st[u].ptr = pp;
            if (pp >= 0) {
#pragma unroll
                for (int w = 0; w < 4; ++w) st[u].m[w] |= sM[pp * 4 + w];
                st[u].s += sS[pp];
                st[u].len += sLen[pp];
                st[u].ptr = sPtr[pp];
            }
        }
        group_sync(1, 128);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = t + 128 * u;
            if (i >= T) continue;
#pragma unroll
            for (int w = 0; w < 4; ++w) sM[i * 4 + w] = st[u].m[w];
            sS[i] = st[u].s;
            sLen[i] = st[u].len;
            sPtr[i] = st[u].ptr;
        }
        group_sync(1, 128);
    }
}

__device__ __forceinline__ void load_k_tile(uint8_t* sm, const CUtensorMap* tmK, uint64_t* bar, int slot, int s,
                                            int hk, int b) {
    mbar_expect_tx(bar, Smem::KS_TILE);
    tma_load_4d(sm + Smem::KS + slot * Smem::KS_TILE, tmK, bar, 0, hk, TP * s, b);
    tma_load_4d(sm + Smem::KS + slot * Smem::KS_TILE + 8192, tmK, bar, 64, hk, TP * s, b);
}

__device__ __forceinline__ void load_qk_tile(uint8_t* sm, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                             uint64_t* bar, int r, int hk, int b) {
    mbar_expect_tx(bar, 4 * TP * 64 * 2);
    tma_load_4d(sm + Smem::QK + 0, tmQ, bar, 0, hk, TP * r, b);
    tma_load_4d(sm + Smem::QK + 16384, tmQ, bar, 64, hk, TP * r, b);
    tma_load_4d(sm + Smem::QK + 8192, tmK, bar, 0, hk, TP * r, b);
    tma_load_4d(sm + Smem::QK + 24576, tmK, bar, 64, hk, TP * r, b);
}

__global__ void __launch_bounds__(NT, 1)
    verify_big_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmS,
                      const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmU, Params p) {
    using L = Smem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* sPar = reinterpret_cast<int*>(sm + L::PAR);
    int* sLen = reinterpret_cast<int*>(sm + L::LEN);
    float* sL2 = reinterpret_cast<float*>(sm + L::L2);
    float* sGam = reinterpret_cast<float*>(sm + L::GAM);
    float* sBeta = reinterpret_cast<float*>(sm + L::BETA);
    double* sLsum = reinterpret_cast<double*>(sm + L::LSUM);
    uint64_t* sMask = reinterpret_cast<uint64_t*>(sm + L::MASK);
    uint8_t* sPath = sm + L::PLIST;
    int* sNin = reinterpret_cast<int*>(sm + L::NIN);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + L::TMEMSLOT);
    volatile int* sFlag = reinterpret_cast<volatile int*>(sm + L::FLAG);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;   // TMEM lane quadrant of this warp
    const int h = blockIdx.x, b = blockIdx.y;
    const int Ts = p.T, H = p.H;  // Ts: the stride of every [B][T] array
    int lbad = 0;
    const int T = stream_len(p.lengths, b, Ts, &lbad);  // this stream's nodes
    const int nb = (T + TP - 1) / TP;                   // its 64-node blocks
    const int hk = h / p.ratio;

    // Nothing global is touched before the preceding kernel of the stream has
    // completed; the next kernel may begin its launch at once.
    pdl_wait();
    pdl_trigger();

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        *sFlag = 0;
        // block 0's Q/K and V tiles and S0 boxes 0 and 1 are requested first,
        // so that they travel while the tree is prepared
        if (nb > 0) {
            load_qk_tile(sm, &tmQ, &tmK, &bars[BAR_QK], 0, hk, b);
            mbar_expect_tx(&bars[BAR_V], 2 * L::V_TILE);
            tma_load_4d(sm + L::VT, &tmV, &bars[BAR_V], 0, h, 0, b);
            tma_load_4d(sm + L::VT + L::V_TILE, &tmV, &bars[BAR_V], 64, h, 0, b);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_expect_tx(&bars[BAR_S0 + i], L::S0_BOX);
            tma_load_4d(sm + L::RX + i * L::S0_BOX, &tmS, &bars[BAR_S0 + i], 32 * i, 0, h, b);
        }
    }
    if (warp == 0) {
        tmem_alloc(sTmem, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();  // barrier initialisation and the tensor-memory address are visible
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);

    if (warp < 4) {
        // ---- tree prep by the solve warps (their named barrier), while the
        // state warps convert S0 and the issuer starts the first Gram
        // product: parents and gates, two nodes per thread (padded nodes
        // have no path, beta 0 and gamma 1), then path bitmasks and
        // root-path log2 gate sums (fp64) by pointer jumping; every CTA of
        // the stream does the same small work ----
        int bad = (tid == 0) ? lbad : 0;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = tid + 128 * u;
            int par = -1;
            float ga = 1.f, gb = 0.f;
            if (i < T) {
                par = p.parent[size_t(b) * Ts + i];
                ga = p.g[(size_t(b) * Ts + i) * H + h];
                gb = p.beta[(size_t(b) * Ts + i) * H + h];
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
            sLsum[i] = (i < T) ? double(log2f(ga)) : 0.0;
            sBeta[i] = gb;
        }
        group_sync(1, 128);
        jump_paths_solve(T, sPar, sLen, sLsum, sMask);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = tid + 128 * u;
            if (i >= T) {
#pragma unroll
                for (int w = 0; w < 4; ++w) sMask[i * 4 + w] = 0ull;
                sLen[i] = 0;
            }
            const float l2 = (i < T) ? float(sLsum[i]) : 0.f;
            sL2[i] = l2;
            sGam[i] = exp2f(l2);
        }
        group_sync(1, 128);
        // tree outputs for the commit: l (natural log), depth, strict-ancestor mask
        if (bad) raise_err(p.err, bad);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = tid + 128 * u;
            if (i >= T) continue;
            p.l[(size_t(b) * Ts + i) * H + h] = sL2[i] * 0.69314718055994531f;
            if (h == 0) {
                p.depth[size_t(b) * Ts + i] = sLen[i] - 1;
                for (int w = 0; w < p.W; ++w) {
                    uint32_t word = uint32_t(sMask[i * 4 + (w >> 1)] >> (32 * (w & 1)));
                    if (w == (i >> 5)) word &= ~(1u << (i & 31));
                    p.mask[(size_t(b) * Ts + i) * p.W + w] = word;
                }
            }
        }
        group_sync(1, 128);  // the tree-prep arrays inside the path lists are no longer read
        if (tid == 0) mbar_arrive(&bars[BAR_PREP]);  // gamma, beta and the masks are ready
    }

    const uint32_t aQK = smem_u32(sm + L::QK);
    uint32_t ks_issued[2] = {0u, 0u};  // issuer: K_s copies per slot

    if (warp == ISSUER / 32) {
        // ================= issuer: Gram tiles, K_s copies, cross terms =================
        if (lane == 0) {
            uint32_t ks_waits[2] = {0u, 0u};
#pragma unroll 1
            for (int r = 0; r < nb; ++r) {
                const uint32_t k_base = uint32_t(r * (r - 1) / 2);  // cross terms before this block
                // the Gram columns are free once the previous block's output
                // product has completed (and so has every earlier product)
                if (r > 0) wait_or_flag(&bars[BAR_W], uint32_t(r - 1) & 1u, sFlag);
                wait_or_flag(&bars[BAR_QK], uint32_t(r) & 1u, sFlag);
                tc_fence_after();
                issue_gram(tmem, aQK, aQK + 8192, 16384);  // (r, r)
                mma_commit(&bars[BAR_G]);
                for (int s = 0; s < 2 && s < r; ++s) {
                    load_k_tile(sm, &tmK, &bars[BAR_KS0 + s], s, s, hk, b);
                    ++ks_issued[s];
                }
                wait_or_flag(&bars[BAR_DREAD], uint32_t(r) & 1u, sFlag);  // the diagonal tile has been read
                if (r > 0) {
                    wait_or_flag(&bars[BAR_KS0], ks_waits[0] & 1u, sFlag);
                    ++ks_waits[0];
                    tc_fence_after();
                    issue_gram(tmem, aQK, smem_u32(sm + L::KS), 8192);  // (r, 0)
                    mma_commit(&bars[BAR_G]);
                }
#pragma unroll 1
                for (int s = 0; s < r; ++s) {
                    const uint32_t k = k_base + uint32_t(s);
                    const int buf = int(k & 1u);
                    wait_or_flag(&bars[BAR_TREAD], k & 1u, sFlag);  // tile s has been read
                    if (s + 2 < r) {  // tile s's Gram product has completed: the next K tile into its slot
                        load_k_tile(sm, &tmK, &bars[BAR_KS0 + (s & 1)], s & 1, s + 2, hk, b);
                        ++ks_issued[s & 1];
                    }
                    if (s + 1 < r) {
                        const int nslot = (s + 1) & 1;
                        wait_or_flag(&bars[BAR_KS0 + nslot], ks_waits[nslot] & 1u, sFlag);
                        ++ks_waits[nslot];
                        tc_fence_after();
                        issue_gram(tmem, aQK, smem_u32(sm + L::KS + nslot * L::KS_TILE), 8192);  // (r, s + 1)
                        mma_commit(&bars[BAR_G]);
                    }
                    wait_or_flag(&bars[BAR_CGB0 + buf], (k >> 1) & 1u, sFlag);  // [C; -G] of tile s is built
                    wait_or_flag(&bars[BAR_XT], uint32_t(r) & 1u, sFlag);  // D holds this block's transformed X
                    tc_fence_after();
                    const uint32_t bH = smem_u32(sm + L::CG + buf * L::CG_BUF), bL = bH + 16384;
#pragma unroll 1
                    for (int pass = 0; pass < 3; ++pass) {  // hi*hi, hi*lo, lo*hi
                        const uint32_t acol = TU + 64 * s + (pass == 2 ? 32 : 0);
                        const uint32_t bb = pass == 1 ? bL : bH;
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16_ts(tmem + TD, tmem + acol + ks * 8, sdesc_sw128(bb + ks * 32),
                                        idesc_bf16(128, 128), 1);
                    }
                    mma_commit(&bars[BAR_CR0 + buf]);
                }
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ================= solve warps: W/M rows, [C; -G] rows =================
        const int rho = tid;              // TMEM lane: Q row rho, or K row rho - 64 of the block
        const bool qrow = rho < TP;
        const int e = rho & (TP - 1);
        float* sX = reinterpret_cast<float*>(sm + L::XV);
        float* sGp = reinterpret_cast<float*>(sm + L::GP);
        float raw[TP];
#pragma unroll 1
        for (int r = 0; r < nb; ++r) {
            const int n0 = TP * r, i = n0 + e;
            const uint32_t g_base = uint32_t(r * (r + 1) / 2);   // Gram commits before this block
            const uint32_t k_base = uint32_t(r * (r - 1) / 2);   // cross terms before this block
            // [M; W] and region X are free once the previous block's output
            // product has completed
            if (r > 0) wait_or_flag(&bars[BAR_W], uint32_t(r - 1) & 1u, sFlag);
            // in-block paths of block r (ascending local index, root side first)
            if (tid < TP) {
                int d = 0;
                for (uint64_t bits = sMask[(n0 + tid) * 4 + r]; bits; bits &= bits - 1)
                    sPath[tid * TP + d++] = uint8_t(__ffsll(static_cast<long long>(bits)) - 1);
                sNin[tid] = d;
            }
            const float li = sL2[i];
            const float bi = sBeta[i];
            wait_or_flag(&bars[BAR_G], g_base & 1u, sFlag);
            tc_fence_after();
            read_gram_row(lane_base, raw);
            tc_fence_before();
            group_sync(1, 128);
            if (tid == 0) {
                mbar_arrive(&bars[BAR_DREAD]);
                if (r == 0) mbar_arrive(&bars[BAR_TGF]);  // no cross terms: the Gram columns are free
            }
            if (r == 0) wait_or_flag(&bars[BAR_SFREE], 0, sFlag);  // the tables overlay the S0 staging

            // ---- W_rr and M_rr rows: C row (Q lanes) or G row (K lanes, strict
            // ancestors, times beta) by in-block path position, then
            // right-looking substitution along path(i): the group of positions
            // 4G..4G+3 is resolved in registers, then applied to the groups
            // below; Gp rows are zero from their own position for four entries,
            // and pivots past the path count as zero ----
            float* xr = sX + rho * XS;
            const int n = sNin[e];
            const uint8_t* pl = sPath + e * TP;
            {
                const int cnt = qrow ? n : n - 1;
                float* dst = qrow ? xr : sGp + e * XS;
                const float sc = qrow ? 1.f : bi;
                for (int d0 = 0; d0 < cnt; d0 += 8) {
                    int jj[8];
                    float rv[8], lv[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) jj[u] = pl[min(d0 + u, cnt - 1)];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        rv[u] = raw[jj[u]];
                        lv[u] = sL2[n0 + jj[u]];
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (d0 + u < cnt) dst[d0 + u] = sc * exp2f(li - lv[u]) * rv[u];
                }
                if (!qrow && n > 0) {
#pragma unroll
                    for (int z = 0; z < 4; ++z) dst[n - 1 + z] = 0.f;
                    for (int d = 0; d < n; ++d) xr[d] = (d == n - 1) ? 1.f : 0.f;
                }
            }
            group_sync(1, 128);
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
                        const float4 gq = *reinterpret_cast<const float4*>(sGp + a[q] * XS + base);
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
                    const float* g0 = sGp + a[0] * XS;
                    const float* g1 = sGp + a[1] * XS;
                    const float* g2 = sGp + a[2] * XS;
                    const float* g3 = sGp + a[3] * XS;
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
                            xg = x4;
                        else
                            *reinterpret_cast<float4*>(xr + 4 * g) = x4;
                    }
                    --G;
                }
            }
            // [scale M_rr; W_rr] row rho -> B operand (K-major bf16, 128-byte swizzle)
            {
                uint8_t* bh = sm + L::MWH + rho * 128;
                uint8_t* bl = sm + L::MWL + rho * 128;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    *reinterpret_cast<uint4*>(bh + ((c8 ^ (rho & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(bl + ((c8 ^ (rho & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                }
                const float msc = qrow ? p.scale : 1.f;  // M rows carry the scale on q
                for (int d = 0; d < n; ++d) {
                    const int j = pl[d];
                    const float x = msc * xr[d];
                    const uint32_t hb = hi_bits(x);
                    const int off = (((j >> 3) ^ (rho & 7)) << 4) + ((j & 7) << 1);
                    *reinterpret_cast<uint16_t*>(bh + off) = uint16_t(hb >> 16);
                    *reinterpret_cast<uint16_t*>(bl + off) = uint16_t(__float_as_uint(x - __uint_as_float(hb)) >> 16);
                }
            }
            fence_proxy_async_smem();
            group_sync(1, 128);  // also: every table read is done before [C; -G] overlays them
            if (tid == 0) mbar_arrive(&bars[BAR_MW]);

            // ---- cross-block terms: rows of [scale C_rs; -G_rs] for s < r; only the
            // entries on root paths are computed (j in block s is on path(i) iff
            // it is a strict ancestor, j < 64 r <= i; decay 2^(l2_i - l2_j) <= 1) ----
            const float rsc = qrow ? p.scale : -bi;
#pragma unroll 1
            for (int s = 0; s < r; ++s) {
                const uint32_t k = k_base + uint32_t(s);   // running index of the cross term
                const int buf = int(k & 1u);
                wait_or_flag(&bars[BAR_G], (g_base + 1 + uint32_t(s)) & 1u, sFlag);
                tc_fence_after();
                read_gram_row(lane_base, raw);
                tc_fence_before();
                group_sync(1, 128);
                if (tid == 0) {
                    mbar_arrive(&bars[BAR_TREAD]);
                    if (s == r - 1) mbar_arrive(&bars[BAR_TGF]);  // the block's last Gram tile has been read
                }
                // buffer buf is free once cross term k - 2 has completed
                if (k >= 2) wait_or_flag(&bars[BAR_CR0 + buf], ((k >> 1) - 1) & 1u, sFlag);
                uint8_t* rh = sm + L::CG + buf * L::CG_BUF + rho * 128;
                uint8_t* rl = rh + 16384;
                const uint64_t bits0 = sMask[i * 4 + s];
                if (__popcll(bits0) > 12) {
                    // many path entries (deep trees): every column in turn
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        float v8[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int jj = 8 * c8 + u;
                            v8[u] = ((bits0 >> jj) & 1ull) ? rsc * exp2f(li - sL2[TP * s + jj]) * raw[jj] : 0.f;
                        }
                        uint4 hv, lv;
                        split2(v8[0], v8[1], hv.x, lv.x);
                        split2(v8[2], v8[3], hv.y, lv.y);
                        split2(v8[4], v8[5], hv.z, lv.z);
                        split2(v8[6], v8[7], hv.w, lv.w);
                        *reinterpret_cast<uint4*>(rh + ((c8 ^ (rho & 7)) << 4)) = hv;
                        *reinterpret_cast<uint4*>(rl + ((c8 ^ (rho & 7)) << 4)) = lv;
                    }
                } else {
                    // few path entries: a zero row, then the entries one by one
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        *reinterpret_cast<uint4*>(rh + ((c8 ^ (rho & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4*>(rl + ((c8 ^ (rho & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                    }
                    for (uint64_t bits = bits0; bits; bits &= bits - 1) {
                        const int jj = __ffsll(static_cast<long long>(bits)) - 1;
                        const float x = rsc * exp2f(li - sL2[TP * s + jj]) * raw[jj];
                        const uint32_t hb = hi_bits(x);
                        const int off = (((jj >> 3) ^ (rho & 7)) << 4) + ((jj & 7) << 1);
                        *reinterpret_cast<uint16_t*>(rh + off) = uint16_t(hb >> 16);
                        *reinterpret_cast<uint16_t*>(rl + off) =
                            uint16_t(__float_as_uint(x - __uint_as_float(hb)) >> 16);
                    }
                }
                fence_proxy_async_smem();
                group_sync(1, 128);
                if (tid == 0) mbar_arrive(&bars[BAR_CGB0 + buf]);
            }
        }
    } else {
        // ================= state warps: S0, X, R', output product, stores =================
        const int c = quad * 32 + lane;  // value column (TMEM lane)
        // S0 rows -> bf16 hi/lo A operand (four boxes through two staging
        // slots, each slot requested again once read)
#pragma unroll 1
        for (int bx = 0; bx < 4; ++bx) {
            const int slot = bx & 1;
            wait_or_flag(&bars[BAR_S0 + slot], uint32_t(bx >> 1), sFlag);
            const uint8_t* rowp = sm + L::RX + slot * L::S0_BOX + c * 128;
            uint32_t wh[16], wl[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 f = *reinterpret_cast<const float4*>(rowp + ((j ^ (c & 7)) << 4));
                split2(f.x, f.y, wh[2 * j], wl[2 * j]);
                split2(f.z, f.w, wh[2 * j + 1], wl[2 * j + 1]);
            }
            tmem_st16(lane_base + TA + bx * 16, wh);
            tmem_st16(lane_base + TA + 64 + bx * 16, wl);
            tmem_wait_st();
            tc_fence_before();
            group_sync(2, 128);
            if (tid == 128) {
                if (bx < 2) {
                    mbar_expect_tx(&bars[BAR_S0 + slot], L::S0_BOX);
                    tma_load_4d(sm + L::RX + slot * L::S0_BOX, &tmS, &bars[BAR_S0 + slot], 32 * (bx + 2), 0, h, b);
                }
                if (bx == 3) mbar_arrive(&bars[BAR_SFREE]);  // the staging area is free
            }
        }
        __syncwarp();
        const uint8_t* vt = sm + L::VT + (c >> 6) * L::V_TILE;
        const int cb = (c & 63) >> 3, cw = (c & 7) << 1;
#pragma unroll 1
        for (int r = 0; r < nb; ++r) {
            const uint32_t pr = uint32_t(r) & 1u;
            const int n0 = TP * r;
            // ---- X = S0 [Q_r; K_r]^T (issued here for block 0, by the previous
            // block's epilogue otherwise), then D <- (scale gamma X_Q | beta (V - gamma X_K)) ----
            if (tid == 128 && r == 0) {
                wait_or_flag(&bars[BAR_QK], pr, sFlag);
                tc_fence_after();
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t db = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                        mma_bf16_ts(tmem + TD, tmem + TA + part * 64 + ks * 8, db, idesc_bf16(128, 128),
                                    (part | ks) != 0);
                    }
                mma_commit(&bars[BAR_X]);
            }
            __syncwarp();
            wait_or_flag(&bars[BAR_X], pr, sFlag);
            wait_or_flag(&bars[BAR_V], pr, sFlag);
            if (r == 0) wait_or_flag(&bars[BAR_PREP], 0, sFlag);  // gamma and beta
            tc_fence_after();
#pragma unroll 1
            for (int hb = 0; hb < 2; ++hb) {
                uint32_t xq[32], xk[32];
                tmem_ld16(lane_base + TD + hb * 32, *reinterpret_cast<uint32_t(*)[16]>(xq));
                tmem_ld16(lane_base + TD + hb * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(xq + 16));
                tmem_ld16(lane_base + TD + 64 + hb * 32, *reinterpret_cast<uint32_t(*)[16]>(xk));
                tmem_ld16(lane_base + TD + 64 + hb * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(xk + 16));
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int el = hb * 32 + e, i = n0 + el;
                    const float gm = sGam[i], be = sBeta[i];
                    const float vv = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16*>(vt + el * 128 + ((cb ^ (el & 7)) << 4) + cw));
                    xq[e] = __float_as_uint(p.scale * gm * __uint_as_float(xq[e]));
                    // nodes past the stream's length are exactly zero (their rows may hold anything)
                    xk[e] = (i < T) ? __float_as_uint(be * (vv - gm * __uint_as_float(xk[e]))) : 0u;
                }
                tmem_st16(lane_base + TD + hb * 32, *reinterpret_cast<uint32_t(*)[16]>(xq));
                tmem_st16(lane_base + TD + hb * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(xq + 16));
                tmem_st16(lane_base + TD + 64 + hb * 32, *reinterpret_cast<uint32_t(*)[16]>(xk));
                tmem_st16(lane_base + TD + 64 + hb * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(xk + 16));
            }
            tmem_wait_st();
            tc_fence_before();
            group_sync(2, 128);
            if (tid == 128) {
                mbar_arrive(&bars[BAR_XT]);
                if (r + 1 < nb) {  // V_r has been read: the next block's V tile
                    mbar_expect_tx(&bars[BAR_V], 2 * L::V_TILE);
                    tma_load_4d(sm + L::VT, &tmV, &bars[BAR_V], 0, h, TP * (r + 1), b);
                    tma_load_4d(sm + L::VT + L::V_TILE, &tmV, &bars[BAR_V], 64, h, TP * (r + 1), b);
                }
            }
            __syncwarp();
            // ---- R' once every cross-block term is in D and the Gram columns are free ----
            wait_or_flag(&bars[BAR_TGF], pr, sFlag);
            if (r > 0) {
                const uint32_t kl = uint32_t(r * (r - 1) / 2 + r - 1);  // the block's last cross term
                wait_or_flag(&bars[BAR_CR0 + (kl & 1u)], (kl >> 1) & 1u, sFlag);
            }
            tc_fence_after();
            // every product that reads Q_r/K_r has completed: the next block's tile
            if (tid == 128 && r + 1 < nb) load_qk_tile(sm, &tmQ, &tmK, &bars[BAR_QK], r + 1, hk, b);
            // R'^T -> bf16 hi/lo in the Gram columns; the K half of D is cleared
            // so that one N = 128 product chain fills both halves
#pragma unroll 1
            for (int hb = 0; hb < 2; ++hb) {
                uint32_t x[32];
                tmem_ld16(lane_base + TD + 64 + hb * 32, *reinterpret_cast<uint32_t(*)[16]>(x));
                tmem_ld16(lane_base + TD + 64 + hb * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(x + 16));
                tmem_wait_ld();
                uint32_t wh[16], wl[16], z[16];
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) {
                    split2(__uint_as_float(x[2 * e2]), __uint_as_float(x[2 * e2 + 1]), wh[e2], wl[e2]);
                    z[e2] = 0u;
                }
                tmem_st16(lane_base + TG + hb * 16, wh);
                tmem_st16(lane_base + TG + 32 + hb * 16, wl);
                tmem_st16(lane_base + TD + 64 + hb * 32, z);
                tmem_st16(lane_base + TD + 64 + hb * 32 + 16, z);
            }
            tmem_wait_st();
            tc_fence_before();
            group_sync(2, 128);
            if (tid == 128) {
                // D += R'^T [scale M_rr; W_rr]^T (bf16 x3): the Q half gains M R', the
                // cleared K half becomes U_r
                wait_or_flag(&bars[BAR_MW], pr, sFlag);
                tc_fence_after();
                const uint32_t bH = smem_u32(sm + L::MWH), bL = smem_u32(sm + L::MWL);
#pragma unroll 1
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t acol = TG + (pass == 2 ? 32 : 0);
                    const uint32_t bb = pass == 1 ? bL : bH;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ts(tmem + TD, tmem + acol + ks * 8, sdesc_sw128(bb + ks * 32), idesc_bf16(128, 128),
                                    1);
                }
                mma_commit(&bars[BAR_W]);
            }
            __syncwarp();
            // ---- U (K half) and o (Q half) by bulk tensor stores of 32-node tiles
            // through the two staging buffers (rows past T are not written).  The
            // U tiles are staged and the o half is held in registers before the
            // next block's X product is issued into D; U_r^T also goes to tensor
            // memory as bf16 hi/lo for the later blocks ----
            wait_or_flag(&bars[BAR_W], pr, sFlag);
            tc_fence_after();
            const bool keep_u = r + 1 < nb;
            // a tile goes by bulk store if it lies inside the stream (or the
            // stream runs to T, where the tensor's bound clips it); a tile the
            // stream ends inside is written from registers, row by row
            const size_t rstride = size_t(H) * DV;
            const size_t obase = (size_t(b) * Ts * H + h) * DV + c;
            bool bulk[2];
            int rows[2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                rows[half] = min(32, T - (n0 + 32 * half));
                bulk[half] = rows[half] == 32 || (T == Ts && rows[half] > 0);
            }
            if (tid == 128) bulk_wait_read<0>();  // the previous block's stores have read the staging tiles
            group_sync(2, 128);
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t y[32];
                tmem_ld16(lane_base + TD + 64 + half * 32, *reinterpret_cast<uint32_t(*)[16]>(y));
                tmem_ld16(lane_base + TD + 64 + half * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(y + 16));
                tmem_wait_ld();
                if (bulk[half]) {
                    float* st = reinterpret_cast<float*>(sm + L::ST + half * L::ST_BUF) + c;
#pragma unroll
                    for (int e = 0; e < 32; ++e) st[e * DV] = __uint_as_float(y[e]);
                } else {
                    float* up = p.U + obase + size_t(n0 + 32 * half) * rstride;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (e < rows[half]) up[e * rstride] = __uint_as_float(y[e]);
                }
                if (keep_u) {
                    uint32_t wh[16], wl[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2)
                        split2(__uint_as_float(y[2 * e2]), __uint_as_float(y[2 * e2 + 1]), wh[e2], wl[e2]);
                    tmem_st16(lane_base + TU + 64 * r + half * 16, wh);
                    tmem_st16(lane_base + TU + 64 * r + 32 + half * 16, wl);
                }
            }
            uint32_t yo[2][32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld16(lane_base + TD + half * 32, *reinterpret_cast<uint32_t(*)[16]>(&yo[half][0]));
                tmem_ld16(lane_base + TD + half * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&yo[half][16]));
            }
            tmem_wait_ld();
            if (keep_u) tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            group_sync(2, 128);  // D has been read and the U tiles are staged
            if (tid == 128) {
                if (bulk[0]) tma_store_4d(&tmU, sm + L::ST, 0, h, n0, b);
                if (bulk[1]) tma_store_4d(&tmU, sm + L::ST + L::ST_BUF, 0, h, n0 + 32, b);
                bulk_commit();
                if (r + 1 < nb) {
                    // the next block's X = S0 [Q; K]^T
                    wait_or_flag(&bars[BAR_QK], pr ^ 1u, sFlag);
                    tc_fence_after();
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint64_t db = sdesc_sw128(aQK + (ks >> 2) * 16384 + (ks & 3) * 32);
                            mma_bf16_ts(tmem + TD, tmem + TA + part * 64 + ks * 8, db, idesc_bf16(128, 128),
                                        (part | ks) != 0);
                        }
                    mma_commit(&bars[BAR_X]);
                }
                bulk_wait_read<0>();  // the U stores have read the staging tiles
            }
            group_sync(2, 128);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint8_t* stg = sm + L::ST + half * L::ST_BUF;
                if (!bulk[half]) {
                    const size_t orow = obase + size_t(n0 + 32 * half) * rstride;
                    if (p.o_bf16) {
                        __nv_bfloat16* op = static_cast<__nv_bfloat16*>(p.o) + orow;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e < rows[half]) op[e * rstride] = __float2bfloat16_rn(__uint_as_float(yo[half][e]));
                    } else {
                        float* op = static_cast<float*>(p.o) + orow;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e < rows[half]) op[e * rstride] = __uint_as_float(yo[half][e]);
                    }
                } else if (p.o_bf16) {
                    __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(stg) + c;
#pragma unroll
                    for (int e = 0; e < 32; ++e) st[e * DV] = __float2bfloat16_rn(__uint_as_float(yo[half][e]));
                } else {
                    float* st = reinterpret_cast<float*>(stg) + c;
#pragma unroll
                    for (int e = 0; e < 32; ++e) st[e * DV] = __uint_as_float(yo[half][e]);
                }
            }
            fence_proxy_async_smem();
            group_sync(2, 128);
            if (tid == 128) {
                if (bulk[0]) tma_store_4d(&tmO, sm + L::ST, 0, h, n0, b);
                if (bulk[1]) tma_store_4d(&tmO, sm + L::ST + L::ST_BUF, 0, h, n0 + 32, b);
                bulk_commit();
            }
        }
        if (tid == 128) bulk_wait<0>();  // every store has completed
    }

    __syncthreads();
    if (*sFlag) {
        // a wait gave up: let the copies and products in flight finish (the
        // latest phase of each barrier, bounded) before leaving
        if (tid == ISSUER) {
            raise_err(p.err, CANOPY_DEVERR_TIMEOUT);
            for (int j = 0; j < 2; ++j)
                if (ks_issued[j]) mbar_wait(&bars[BAR_KS0 + j], (ks_issued[j] - 1) & 1u);
            const uint32_t ng = uint32_t(nb * (nb + 1) / 2), nk = uint32_t(nb * (nb - 1) / 2);
            mbar_wait(&bars[BAR_G], (ng - 1) & 1u);
            if (nk > 0) mbar_wait(&bars[BAR_CR0], (((nk + 1) >> 1) - 1) & 1u);
            if (nk > 1) mbar_wait(&bars[BAR_CR1], ((nk >> 1) - 1) & 1u);
        }
        if (tid == 128) {
            mbar_wait(&bars[BAR_S0], 1);
            mbar_wait(&bars[BAR_S0B], 1);
            mbar_wait(&bars[BAR_QK], uint32_t(nb - 1) & 1u);
            mbar_wait(&bars[BAR_V], uint32_t(nb - 1) & 1u);
            mbar_wait(&bars[BAR_X], uint32_t(nb - 1) & 1u);
            mbar_wait(&bars[BAR_W], uint32_t(nb - 1) & 1u);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace tcb

// ---------------------------------------------------------------------------
// Host side.

bool make_bf16_row_map(CUtensorMap* m, const void* base, int B, int T, int H);
bool make_state_map(CUtensorMap* m, const float* base, int B, int H);
bool make_row_store_map(CUtensorMap* m, void* base, int bf16, int B, int T, int H);

cudaError_t launch_verify_tc_big(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const float* S0, const int32_t* parent, const int32_t* lengths, int T, int B, int H,
                                 int HK, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st) {
    if (T <= tcb::TP || T > kMaxT) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, ms, mo, mu;
    if (!make_bf16_row_map(&mq, q, B, T, HK) || !make_bf16_row_map(&mk, k, B, T, HK) ||
        !make_bf16_row_map(&mv, v, B, T, H) || !make_state_map(&ms, S0, B, H) ||
        !make_row_store_map(&mo, o, o_bf16, B, T, H) || !make_row_store_map(&mu, ws.U, 0, B, T, H))
        return cudaErrorInvalidValue;
    tcb::Params prm;
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
    const int smem = tcb::Smem::TOTAL + 1024;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(tcb::verify_big_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    return launch_pdl(tcb::verify_big_kernel, dim3(H, B), dim3(tcb::NT), smem, st, mq, mk, mv, ms, mo, mu, prm);
}

}  // namespace canopy
