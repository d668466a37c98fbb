// Tree preparation kernel: parent array -> validation, depth, strict-ancestor
// bitmask, DFS pre-order, and cumulative log gates l for every head.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form"
// (A(i), path(i), depth, l_i = log alpha_i + l_parent(i)) and "Design
// decisions" (DFS pre-order keeps subtrees contiguous; a T x T bitmask).
// One CTA of 256 threads per (stream, group of HC heads); T <= 256.
#include "common.cuh"

namespace canopy {

namespace prep {

constexpr int HC = 4;  // heads per CTA

__global__ void __launch_bounds__(256) tree_prep_kernel(const int32_t* __restrict__ parent,
                                                        const int32_t* __restrict__ lengths,
                                                        const float* __restrict__ g, int Ts, int H, Ws ws,
                                                        int with_order) {
    __shared__ int sPtr[kMaxT];
    __shared__ int sLen[kMaxT];
    __shared__ int sPar[kMaxT];
    __shared__ float sS[kMaxT];
    __shared__ uint64_t sM[kMaxT * 4];
    __shared__ int sSize[kMaxT];
    __shared__ int sPos[kMaxT];
    __shared__ double sLg[kMaxT * HC];  // log gates, then cumulative sums, for HC heads (summed in
                                        // fp64: l_i - l_j must stay accurate over deep paths)
    __shared__ int sJp[kMaxT];         // jump pointers
    const int b = blockIdx.x, i = threadIdx.x;
    const int hc = blockIdx.y;            // this CTA's HC heads
    const bool lead = hc == 0;            // writes the per-stream outputs
    // Ts is the stride of every [B][T] array, T this stream's node count
    // (nodes past it are neither read nor written)
    int lbad = 0;
    const int T = stream_len(lengths, b, Ts, &lbad);
    if (lbad && lead && i == 0) raise_err(ws.err, lbad);
    int bad = 0;
    if (i < T) {
        int par = parent[size_t(b) * Ts + i];
        const bool ok = (i == 0) ? (par == -1) : (par >= 0 && par < i);
        if (!ok) {
            bad |= CANOPY_DEVERR_TREE;
            par = (i == 0) ? -1 : 0;
        }
        sPtr[i] = par;
        sPar[i] = par;
        sS[i] = 0.f;
    }
    if (bad && lead) raise_err(ws.err, bad);
    __syncthreads();
    jump_paths<4>(T, sPtr, sLen, sS, sM);

    // depth and strict-ancestor mask
    if (lead && i < T) {
        ws.depth[size_t(b) * Ts + i] = sLen[i] - 1;
        for (int w = 0; w < ws.W; ++w) {
            uint64_t word = sM[i * 4 + (w >> 1)];
            if ((w >> 1) == (i >> 6)) word &= ~(1ull << (i & 63));
            ws.mask[(size_t(b) * Ts + i) * ws.W + w] = uint32_t(word >> (32 * (w & 1)));
        }
    }

    // cumulative log gates l_n = log g_n + l_parent(n) for every head, by
    // pointer jumping over HC heads at a time (ceil(log2 T) rounds)
    int badg = 0;
    for (int h0 = HC * hc; h0 < min(H, HC * hc + HC); h0 += HC) {
        const int hn = min(HC, H - h0);
        __syncthreads();
        for (int e = i; e < T * hn; e += blockDim.x) {
            const int n = e / hn, hh = e % hn;
            float a = g[(size_t(b) * Ts + n) * H + h0 + hh];
            if (!(a > 0.f) || !isfinite(a)) {
                badg = CANOPY_DEVERR_GATE;
                a = 1.f;
            }
            sLg[n * HC + hh] = double(logf(a));  // fp32 log, fp64 sums
        }
        if (i < T) sJp[i] = sPar[i];
        __syncthreads();
        for (int span = 1; span < T; span *= 2) {
            double nv[HC];
            int np = -1;
#pragma unroll
            for (int u = 0; u < HC; ++u) {
                const int e = i + u * 256;
                nv[u] = 0.0;
                if (e < T * hn) {
                    const int n = e / hn, hh = e % hn, pn = sJp[n];
                    nv[u] = sLg[n * HC + hh] + ((pn >= 0) ? sLg[pn * HC + hh] : 0.0);
                }
            }
            if (i < T) np = (sJp[i] >= 0) ? sJp[sJp[i]] : -1;
            __syncthreads();
#pragma unroll
            for (int u = 0; u < HC; ++u) {
                const int e = i + u * 256;
                if (e < T * hn) sLg[(e / hn) * HC + e % hn] = nv[u];
            }
            if (i < T) sJp[i] = np;
            __syncthreads();
        }
        for (int e = i; e < T * hn; e += blockDim.x) {
            const int n = e / hn, hh = e % hn;
            ws.l[(size_t(b) * Ts + n) * H + h0 + hh] = float(sLg[n * HC + hh]);
        }
    }
    if (badg) raise_err(ws.err, badg);

    // DFS pre-order (children in index order): subtree sizes bottom-up, then
    // each child takes the next free slot after its parent.
    __syncthreads();
    if (!lead || !with_order) return;
    if (i == 0) {
        for (int n = 0; n < T; ++n) sSize[n] = 1;
        for (int n = T - 1; n >= 1; --n) sSize[sPar[n]] += sSize[n];
        sPos[0] = 0;
        for (int n = 0; n < T; ++n) sLen[n] = 1;  // reuse: next free offset below n
        for (int n = 1; n < T; ++n) {
            const int pn = sPar[n];
            sPos[n] = sPos[pn] + sLen[pn];
            sLen[pn] += sSize[n];
        }
    }
    __syncthreads();
    if (i < T) ws.order[size_t(b) * Ts + sPos[i]] = i;
}

}  // namespace prep

cudaError_t launch_tree_prep(const int32_t* parent, const int32_t* lengths, const float* g, int T, int B, int H,
                             const Ws& ws, int with_order, cudaStream_t st) {
    const dim3 grid(B, (H + prep::HC - 1) / prep::HC);
    prep::tree_prep_kernel<<<grid, 256, 0, st>>>(parent, lengths, g, T, H, ws, with_order);
    return cudaGetLastError();
}

}  // namespace canopy
