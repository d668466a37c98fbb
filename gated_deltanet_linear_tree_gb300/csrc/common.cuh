// Shared device/host helpers for libcanopy: workspace layout, error bits,
// bf16 helpers, and inline-PTX wrappers for mbarrier, TMA and tcgen05
// (Blackwell tensor cores with tensor-memory accumulators), sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/canopy.h"

namespace canopy {

// ---------------------------------------------------------------------------
// Workspace layout (see canopy_workspace_bytes in the public header).

struct WsLayout {
    size_t U, l, depth, mask, order, err, gs, cs, xq, rr, total;
    int W;  // 32-bit words per mask row
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline WsLayout ws_layout(int B, int T, int H, int dv) {
    WsLayout w;
    w.W = (T + 31) / 32;
    const size_t BT = size_t(B) * T;
    w.err = 0;  // first, so its offset does not depend on the sizes
    size_t o = 256;
    // tree-prep outputs next: their offsets do not depend on dv
    w.l = o;     o = ws_align(o + BT * H * 4);
    w.depth = o; o = ws_align(o + BT * 4);
    w.mask = o;  o = ws_align(o + BT * w.W * 4);
    w.order = o; o = ws_align(o + BT * 4);
    w.U = o;     o = ws_align(o + BT * H * dv * 4);
    // scratch of the fp32 path: G and C as [B][H][T][T], gamma*Q S0^T and R as [B][T][H][dv]
    w.gs = o;    o = ws_align(o + size_t(B) * H * T * T * 4);
    w.cs = o;    o = ws_align(o + size_t(B) * H * T * T * 4);
    w.xq = o;    o = ws_align(o + BT * H * dv * 4);
    w.rr = o;    o = ws_align(o + BT * H * dv * 4);
    w.total = o;
    return w;
}

struct Ws {
    float* U;
    float* l;
    int32_t* depth;
    uint32_t* mask;
    int32_t* order;
    int32_t* err;
    float* gs;
    float* cs;
    float* xq;
    float* rr;
    int W;
};

inline Ws ws_bind(void* base, int B, int T, int H, int dv) {
    WsLayout L = ws_layout(B, T, H, dv);
    char* p = static_cast<char*>(base);
    Ws w;
    w.U = reinterpret_cast<float*>(p + L.U);
    w.l = reinterpret_cast<float*>(p + L.l);
    w.depth = reinterpret_cast<int32_t*>(p + L.depth);
    w.mask = reinterpret_cast<uint32_t*>(p + L.mask);
    w.order = reinterpret_cast<int32_t*>(p + L.order);
    w.err = reinterpret_cast<int32_t*>(p + L.err);
    w.gs = reinterpret_cast<float*>(p + L.gs);
    w.cs = reinterpret_cast<float*>(p + L.cs);
    w.xq = reinterpret_cast<float*>(p + L.xq);
    w.rr = reinterpret_cast<float*>(p + L.rr);
    w.W = L.W;
    return w;
}

constexpr int kMaxT = 256;

// ---------------------------------------------------------------------------
// Input loads: q/k/v are bf16 or fp32.

template <typename T>
__device__ inline float to_f(T x);
template <>
__device__ inline float to_f<float>(float x) { return x; }
template <>
__device__ inline float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Four consecutive elements starting at p (16-byte aligned for fp32, 8 for bf16).
__device__ inline float4 load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ inline float4 load4(const __nv_bfloat16* p) {
    uint2 r = __ldg(reinterpret_cast<const uint2*>(p));
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&r.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&r.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

__device__ inline void store_out(float* p, float x) { *p = x; }
__device__ inline void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Gate checks shared by every kernel: alpha must be finite and > 0, beta finite.
__device__ inline bool gate_ok(float a, float b) {
    return (a > 0.f) && isfinite(a) && isfinite(b);
}

__device__ inline void raise_err(int32_t* err, int bits) { atomicOr(err, bits); }

// Nodes of stream b in a ragged batch: lengths[b], or T without lengths.  A
// value outside [0, T] is read as the nearest bound and sets
// CANOPY_DEVERR_LENGTH in *bad.
__device__ inline int stream_len(const int32_t* lengths, int b, int T, int* bad) {
    if (!lengths) return T;
    const int n = lengths[b];
    if (n < 0 || n > T) {
        *bad |= CANOPY_DEVERR_LENGTH;
        return n < 0 ? 0 : T;
    }
    return n;
}

// ---------------------------------------------------------------------------
// Bounded waits use the global nanosecond timer.

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ inline unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ inline uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch -----------------------------------------
// A kernel launched with launch_pdl() may start while the previous kernel of
// the stream is still running; pdl_wait() blocks until that kernel has
// completed and its memory is visible (a no-op otherwise), and pdl_trigger()
// lets the next such kernel begin its own launch.  Kernels here call both
// before their first global access, so only launch latency and the previous
// kernel's tail overlap.
__device__ inline void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ inline void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- mbarrier --------------------------------------------------------------

__device__ inline void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ inline void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ inline void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ inline bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Returns false if the phase did not complete within kWaitLimitNs.
__device__ inline bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255) == 255 && globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

__device__ inline void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier among `n` threads (a multiple of 32) of the CTA on named barrier `id`.
__device__ inline void group_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Ask L2 to fetch [p, p + bytes) (16-byte aligned, bytes a multiple of 16).
__device__ inline void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy
// (tensor cores, TMA) before a barrier.
__device__ inline void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA -------------------------------------------------------------------

__device__ inline void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                   int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Tiled bulk store shared -> global through a tensor map (bulk-group
// completion: commit with bulk_commit(), then bulk_wait_read<N>() before the
// shared source is rewritten and bulk_wait<0>() before leaving).  Elements
// outside the tensor are not written.
__device__ inline void tma_store_4d(const CUtensorMap* map, const void* src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}
__device__ inline void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// At most N committed bulk groups of this thread still read their shared source.
template <int N>
__device__ inline void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// At most N committed bulk groups of this thread are still incomplete.
template <int N>
__device__ inline void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Untiled bulk copy global -> shared, completing on `bar` (both addresses
// 16-byte aligned, bytes a multiple of 16).
__device__ inline void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// ---- tcgen05 ---------------------------------------------------------------

__device__ inline void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ inline void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ inline void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ inline void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ inline void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout (rows of 128 bytes, 8-row groups 1024 bytes apart).  The tile base
// must be 1024-byte aligned; a K offset inside the 128-byte row is added to
// the start address.
__device__ inline uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);  // start address, bits 0-13
    d |= uint64_t(1) << 16;                   // leading byte offset (unused here)
    d |= uint64_t(1024 >> 4) << 32;           // stride byte offset: 8 rows x 128 B
    d |= uint64_t(1) << 46;                   // descriptor version for tcgen05
    d |= uint64_t(2) << 61;                   // 128-byte swizzle
    return d;
}

// Instruction descriptors: fp32 accumulate, A and B K-major, dense.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, K = 16.
__device__ inline void mma_bf16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, tf32 inputs, K = 8.
__device__ inline void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, K = 16 (A: 8 columns of
// bf16 pairs per lane, the lower K index in the low half).
__device__ inline void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// Arrive on `bar` when every MMA issued so far by this thread has completed.
__device__ inline void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns per thread.
__device__ inline void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ inline void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// 32 lanes x 32 bits, 8 consecutive columns per thread.
__device__ inline void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
// 16 lanes x 256 bits, 4 repetitions along the columns (32 columns): for
// repetition k, thread t holds r[4k] = (lane t/4, column 8k + 2(t%4)),
// r[4k+1] = the next column, r[4k+2], r[4k+3] = the same columns of lane
// t/4 + 8 (lanes relative to the 16-lane base of the address).
__device__ inline void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ inline void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ inline void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Round an fp32 value to the nearest tf32 (ties away from zero).
__device__ inline uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// ---------------------------------------------------------------------------
// Tree preparation by pointer jumping, for one stream, run by a whole CTA.
//
// canopy page, "The tree closed form": path(i) = A(i) + {i}, depth |A(i)|,
// l_i = log alpha_i + l_parent(i).  Each node keeps (segment mask, segment
// log-gate sum, segment length, jump pointer); a round merges a node's
// segment with its jump target's and doubles the jump, so ceil(log2 T)
// rounds cover every root path.  NW = 64-bit mask words (T <= 64 NW).

template <int NW, typename S = float>
struct JumpState {
    uint64_t m[NW];
    S s;
    int len;
    int ptr;
};

// sPtr/sLen/sS/sM: shared arrays of Tcap entries (sM: Tcap*NW words).  On
// entry sPtr[i] holds the sanitised parent and sS[i] the per-node log gate
// (node i < T); on exit sM holds path(i) (self included), sS the cumulative
// log gate (summed in S: float, or double where deep paths need it) and
// sLen |path(i)|.  Requires blockDim.x >= T.
template <int NW, typename S = float>
__device__ inline void jump_paths(int T, int* sPtr, int* sLen, S* sS, uint64_t* sM) {
    const int i = threadIdx.x;
    if (i < T) {
        for (int w = 0; w < NW; ++w) sM[i * NW + w] = (w == (i >> 6)) ? (1ull << (i & 63)) : 0ull;
        sLen[i] = 1;
    }
    __syncthreads();
    for (int round = 0; round < 9; ++round) {
        int more = 0;
        JumpState<NW, S> st;
        if (i < T) {
            int p = sPtr[i];
            for (int w = 0; w < NW; ++w) st.m[w] = sM[i * NW + w];
            st.s = sS[i];
            st.len = sLen[i];
            st.ptr = p;
            if (p >= 0) {
                for (int w = 0; w < NW; ++w) st.m[w] |= sM[p * NW + w];
                st.s += sS[p];
                st.len += sLen[p];
                st.ptr = sPtr[p];
                more = st.ptr >= 0;
            }
        }
        __syncthreads();
        if (i < T) {
            for (int w = 0; w < NW; ++w) sM[i * NW + w] = st.m[w];
            sS[i] = st.s;
            sLen[i] = st.len;
            sPtr[i] = st.ptr;
        }
        if (!__syncthreads_or(more)) break;
    }
}

}  // namespace canopy
