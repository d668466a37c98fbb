// extern "C" entry points of libcanopy.so: argument checks, workspace
// binding and kernel dispatch.  See include/canopy.h for the contract.
#include <cmath>

#include "common.cuh"

namespace canopy {
int path_replay_max_t();
// Launchers take H = value heads (the units: v, g, beta, S0, o, workspace)
// and HK = key heads (q, k); value head h reads key head h / (H / HK).
cudaError_t launch_tree_prep(const int32_t* parent, const int32_t* lengths, const float* g, int T, int B, int H,
                             const Ws& ws, int with_order, cudaStream_t st);
cudaError_t launch_verify_neumann(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                  const float* S0, const int32_t* parent, int T, int B, int H, int HK, void* o,
                                  int o_bf16, float scale, const Ws& ws, cudaStream_t st);
cudaError_t launch_verify_tc_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const float* S0, const int32_t* parent, const int32_t* lengths, int T, int B, int H,
                                 int HK, void* o, int o_bf16, float scale, const Ws& ws, int inputs_ready,
                                 int state_ready, cudaStream_t st);
cudaError_t launch_verify_tc_big(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const float* S0, const int32_t* parent, const int32_t* lengths, int T, int B, int H,
                                 int HK, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st);
cudaError_t launch_verify_simt(const void* q, const void* k, const void* v, int in_bf16, const float* beta,
                               const float* S0, const int32_t* lengths, int T, int B, int H, int HK, int d, void* o,
                               int o_bf16, float scale, const Ws& ws, cudaStream_t st);
cudaError_t launch_gram_tc(const void* q, const void* k, const void* v, const float* beta, const float* S0, int T,
                           int B, int H, int HK, const Ws& ws, cudaStream_t st);
cudaError_t launch_commit(const int32_t* accepted, const int32_t* parent, const int32_t* lengths, const float* S0,
                          float* S_new, const void* k, int in_bf16, int T, int B, int H, int HK, int d, const Ws& ws,
                          int state_ready, cudaStream_t st);
cudaError_t launch_serial(const void* q, const void* k, const void* v, int in_bf16, const float* g,
                          const float* beta, const float* S0, const int32_t* parent, int T, int B, int H, int HK,
                          int d, void* o, int o_bf16, float scale, float* snap, int32_t* err, cudaStream_t st);
cudaError_t launch_path_replay(const void* q, const void* k, const void* v, int in_bf16, const float* g,
                               const float* beta, const float* S0, const int32_t* parent, const int32_t* lengths,
                               int T, int B, int H, int HK, int d, void* o, int o_bf16, float scale, const Ws& ws,
                               cudaStream_t st);
cudaError_t launch_solve_variant(int variant, int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws,
                                 cudaStream_t st);
cudaError_t launch_tree_conv(const void* x, int bf16, const float* state, const float* w, const float* bias,
                             const int32_t* parent, int T, int B, int C, int K, int silu, void* y, int32_t* err,
                             cudaStream_t st);
cudaError_t launch_conv_commit(const int32_t* accepted, const void* x, int bf16, const int32_t* parent,
                               const float* state, float* state_new, int T, int B, int C, int K, int32_t* err,
                               cudaStream_t st);
}  // namespace canopy

using namespace canopy;

namespace {

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool sizes_ok(int B, int T, int H) { return B >= 1 && H >= 1 && T >= 1 && T <= kMaxT; }

// Dispatch below the crossover (canopy page, "Design decisions": the serial
// path below it, the closed form above): replaying each node's root path
// from S0 beats the closed form's fixed chain of dependent stages for trees
// of one or two nodes, and for three-node trees while there are few (stream,
// value head) pairs to spread over the GPU.  From the GB300 dispatch table
// (profiles/dispatch_H16_d128.jsonl: random trees, 16 value heads, replay /
// closed form time): T = 1: 0.57-0.73; T = 2: 0.64-0.90; T = 3: 0.79-0.95
// up to B = 8, 1.03 at B = 16; T = 4: 0.96-1.03 up to B = 4, 1.10 and more
// beyond; T >= 5: above 1.09.  tests/test_dispatch_table.py checks the rule
// against that table.
bool path_replay_wins(int T, int B, int HV) {
    const size_t units = size_t(B) * HV;
    return T <= 2 || (T == 3 && units <= 128);
}

// key heads H, value heads HV: HV a positive multiple of H
bool heads_ok(int H, int HV) { return H >= 1 && HV >= H && HV % H == 0; }

canopy_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CANOPY_OK : CANOPY_ERR_CUDA; }

constexpr unsigned kVerifyFlags =
    CANOPY_VERIFY_INPUTS_READY | CANOPY_VERIFY_STATE_READY | CANOPY_VERIFY_CLOSED_FORM | CANOPY_VERIFY_PATH_REPLAY;

// The checks of a verify call that do not look at pointers.
canopy_status verify_args(int T, int B, int H, int HV, canopy_dtype in_dtype, canopy_dtype o_dtype, int dk, int dv,
                          canopy_solve solve, unsigned flags, int has_lengths, float scale) {
    if ((in_dtype != CANOPY_F32 && in_dtype != CANOPY_BF16) || (o_dtype != CANOPY_F32 && o_dtype != CANOPY_BF16) ||
        (solve != CANOPY_SOLVE_FWDSUB && solve != CANOPY_SOLVE_NEUMANN && solve != CANOPY_SOLVE_SQUARING &&
         solve != CANOPY_SOLVE_SPLIT) ||
        (flags & ~kVerifyFlags) || !std::isfinite(scale))
        return CANOPY_ERR_ARG;
    const unsigned force = flags & (CANOPY_VERIFY_CLOSED_FORM | CANOPY_VERIFY_PATH_REPLAY);
    if (force == (CANOPY_VERIFY_CLOSED_FORM | CANOPY_VERIFY_PATH_REPLAY) || (force && solve != CANOPY_SOLVE_FWDSUB))
        return CANOPY_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0 || !heads_ok(H, HV)) return CANOPY_ERR_ARG;
    if (!sizes_ok(B, T, HV) || dk != dv || (dk != 128 && dk != 32)) return CANOPY_ERR_UNSUPPORTED;
    const bool bf16_128 = in_dtype == CANOPY_BF16 && dk == 128;
    // the solve variants run on the tensor-core Gram's tiles (bf16, d = 128), uniform T
    if (solve != CANOPY_SOLVE_FWDSUB && (!bf16_128 || has_lengths)) return CANOPY_ERR_UNSUPPORTED;
    if ((flags & CANOPY_VERIFY_PATH_REPLAY) && T > path_replay_max_t()) return CANOPY_ERR_UNSUPPORTED;
    return CANOPY_OK;
}

// The plan of a verify call whose arguments passed verify_args.
canopy_plan verify_plan(int T, int B, int HV, canopy_dtype in_dtype, int dk, canopy_solve solve, unsigned flags) {
    const bool bf16_128 = in_dtype == CANOPY_BF16 && dk == 128;
    if (solve == CANOPY_SOLVE_FWDSUB) {
        if (flags & CANOPY_VERIFY_PATH_REPLAY) return CANOPY_PLAN_PATH_REPLAY;
        if (!(flags & CANOPY_VERIFY_CLOSED_FORM) && path_replay_wins(T, B, HV)) return CANOPY_PLAN_PATH_REPLAY;
        if (bf16_128) return T <= 64 ? CANOPY_PLAN_TC_BLOCK : CANOPY_PLAN_TC_BLOCKED;
        return CANOPY_PLAN_FP32;
    }
    if (solve == CANOPY_SOLVE_NEUMANN && T <= 64) return CANOPY_PLAN_TC_NEUMANN;
    return CANOPY_PLAN_VARIANT;
}

}  // namespace

extern "C" {

size_t canopy_workspace_bytes(int B, int T, int HV, int dk, int dv) {
    if (!sizes_ok(B, T, HV) || dk != dv || (dk != 128 && dk != 32)) return 0;
    return ws_layout(B, T, HV, dv).total;
}

size_t canopy_workspace_offset(int B, int T, int HV, int dk, int dv, canopy_ws_region region) {
    if (canopy_workspace_bytes(B, T, HV, dk, dv) == 0) return ~size_t(0);
    const WsLayout L = ws_layout(B, T, HV, dv);
    switch (region) {
        case CANOPY_WS_ERR: return L.err;
        case CANOPY_WS_L: return L.l;
        case CANOPY_WS_DEPTH: return L.depth;
        case CANOPY_WS_MASK: return L.mask;
        case CANOPY_WS_ORDER: return L.order;
        case CANOPY_WS_U: return L.U;
    }
    return ~size_t(0);
}

canopy_status canopy_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (!aligned16(workspace) || bytes == 0) return CANOPY_ERR_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)));
}

size_t canopy_snapshot_bytes(int B, int T, int HV, int dk, int dv) {
    if (!sizes_ok(B, T, HV) || dk != dv || (dk != 128 && dk != 32)) return 0;
    return size_t(B) * T * HV * dv * dk * 4;
}

canopy_status canopy_tree_prep(const int32_t* parent, const float* g, int T, int B, int HV, void* workspace,
                               void* stream) {
    if (!aligned16(parent) || !aligned16(g) || !aligned16(workspace)) return CANOPY_ERR_ARG;
    if (!sizes_ok(B, T, HV)) return CANOPY_ERR_UNSUPPORTED;
    Ws ws = ws_bind(workspace, B, T, HV, 32);  // tree-prep regions do not depend on dv
    return cuda_status(launch_tree_prep(parent, nullptr, g, T, B, HV, ws, 1, static_cast<cudaStream_t>(stream)));
}

canopy_status canopy_tree_verify(const void* q, const void* k, const void* v, canopy_dtype in_dtype,
                                 const float* g, const float* beta, const float* S0, const int32_t* parent,
                                 const int32_t* lengths, int T, int B, int H, int HV, int dk, int dv, float scale,
                                 canopy_solve solve, void* o, canopy_dtype o_dtype, void* workspace, unsigned flags,
                                 void* stream) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) || !aligned16(S0) ||
        !aligned16(parent) || !aligned16(o) || !aligned16(workspace) || (lengths && !aligned16(lengths)))
        return CANOPY_ERR_ARG;
    const canopy_status as = verify_args(T, B, H, HV, in_dtype, o_dtype, dk, dv, solve, flags, lengths != nullptr,
                                         scale);
    if (as != CANOPY_OK) return as;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws ws = ws_bind(workspace, B, T, HV, dv);
    const int in_bf16 = in_dtype == CANOPY_BF16, o_bf16 = o_dtype == CANOPY_BF16;
    switch (verify_plan(T, B, HV, in_dtype, dk, solve, flags)) {
        case CANOPY_PLAN_PATH_REPLAY:
            return cuda_status(launch_path_replay(q, k, v, in_bf16, g, beta, S0, parent, lengths, T, B, HV, H, dk, o,
                                                  o_bf16, scale, ws, st));
        case CANOPY_PLAN_TC_BLOCK:
            return cuda_status(launch_verify_tc_fwd(q, k, v, g, beta, S0, parent, lengths, T, B, HV, H, o, o_bf16,
                                                    scale, ws, (flags & CANOPY_VERIFY_INPUTS_READY) != 0,
                                                    (flags & CANOPY_VERIFY_STATE_READY) != 0, st));
        case CANOPY_PLAN_TC_NEUMANN:
            return cuda_status(
                launch_verify_neumann(q, k, v, g, beta, S0, parent, T, B, HV, H, o, o_bf16, scale, ws, st));
        case CANOPY_PLAN_TC_BLOCKED:
            return cuda_status(
                launch_verify_tc_big(q, k, v, g, beta, S0, parent, lengths, T, B, HV, H, o, o_bf16, scale, ws, st));
        case CANOPY_PLAN_FP32: {
            const cudaError_t e = launch_tree_prep(parent, lengths, g, T, B, HV, ws, 0, st);
            if (e != cudaSuccess) return CANOPY_ERR_CUDA;
            return cuda_status(
                launch_verify_simt(q, k, v, in_bf16, beta, S0, lengths, T, B, HV, H, dk, o, o_bf16, scale, ws, st));
        }
        case CANOPY_PLAN_VARIANT: {
            // Neumann beyond 64 nodes, squaring and split: tree prep, Gram tiles, then the solve
            cudaError_t e = launch_tree_prep(parent, nullptr, g, T, B, HV, ws, 0, st);
            if (e != cudaSuccess) return CANOPY_ERR_CUDA;
            e = launch_gram_tc(q, k, v, beta, S0, T, B, HV, H, ws, st);
            if (e != cudaSuccess) return cuda_status(e);
            return cuda_status(launch_solve_variant(int(solve), T, B, HV, o, o_bf16, scale, ws, st));
        }
        default:
            return CANOPY_ERR_ARG;
    }
}

canopy_plan canopy_verify_plan(int T, int B, int H, int HV, canopy_dtype in_dtype, int dk, int dv,
                               canopy_solve solve, unsigned flags, int has_lengths) {
    if (verify_args(T, B, H, HV, in_dtype, CANOPY_F32, dk, dv, solve, flags, has_lengths, 1.f) != CANOPY_OK)
        return CANOPY_PLAN_NONE;
    return verify_plan(T, B, HV, in_dtype, dk, solve, flags);
}

canopy_status canopy_commit(const int32_t* accepted, const float* S0, float* S_new, const void* k,
                            const int32_t* parent, const int32_t* lengths, canopy_dtype in_dtype, int T, int B,
                            int H, int HV, int dk, int dv, const void* workspace, unsigned flags, void* stream) {
    if (!aligned16(accepted) || !aligned16(S0) || !aligned16(S_new) || !aligned16(k) || !aligned16(parent) ||
        !aligned16(workspace) || (lengths && !aligned16(lengths)))
        return CANOPY_ERR_ARG;
    if (in_dtype != CANOPY_F32 && in_dtype != CANOPY_BF16) return CANOPY_ERR_ARG;
    if (flags & ~CANOPY_COMMIT_STATE_READY) return CANOPY_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0 || !heads_ok(H, HV)) return CANOPY_ERR_ARG;
    if (!sizes_ok(B, T, HV) || dk != dv || (dk != 128 && dk != 32)) return CANOPY_ERR_UNSUPPORTED;
    Ws ws = ws_bind(const_cast<void*>(workspace), B, T, HV, dv);
    return cuda_status(launch_commit(accepted, parent, lengths, S0, S_new, k, in_dtype == CANOPY_BF16, T, B, HV, H,
                                     dk, ws,
                                     (flags & CANOPY_COMMIT_STATE_READY) != 0, static_cast<cudaStream_t>(stream)));
}

canopy_status canopy_serial_replay(const void* q, const void* k, const void* v, canopy_dtype in_dtype,
                                   const float* g, const float* beta, const float* S0, const int32_t* parent, int T,
                                   int B, int H, int HV, int dk, int dv, float scale, void* o, canopy_dtype o_dtype,
                                   void* snapshot, void* workspace, void* stream) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) || !aligned16(S0) ||
        !aligned16(parent) || !aligned16(o) || !aligned16(snapshot) || !aligned16(workspace))
        return CANOPY_ERR_ARG;
    if ((in_dtype != CANOPY_F32 && in_dtype != CANOPY_BF16) || (o_dtype != CANOPY_F32 && o_dtype != CANOPY_BF16) ||
        !std::isfinite(scale))
        return CANOPY_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0 || !heads_ok(H, HV)) return CANOPY_ERR_ARG;
    if (!sizes_ok(B, T, HV) || dk != dv || (dk != 128 && dk != 32)) return CANOPY_ERR_UNSUPPORTED;
    Ws ws = ws_bind(workspace, B, T, HV, dv);
    return cuda_status(launch_serial(q, k, v, in_dtype == CANOPY_BF16, g, beta, S0, parent, T, B, HV, H, dk, o,
                                     o_dtype == CANOPY_BF16, scale, static_cast<float*>(snapshot), ws.err,
                                     static_cast<cudaStream_t>(stream)));
}

canopy_status canopy_tree_conv(const void* x, canopy_dtype dtype, const float* conv_state, const float* weight,
                               const float* bias, const int32_t* parent, int T, int B, int C, int K,
                               canopy_activation act, void* y, int32_t* err, void* stream) {
    if (!aligned16(x) || !aligned16(conv_state) || !aligned16(weight) || !aligned16(parent) || !aligned16(y) ||
        (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) || (err && (reinterpret_cast<uintptr_t>(err) & 3u)))
        return CANOPY_ERR_ARG;
    if ((dtype != CANOPY_F32 && dtype != CANOPY_BF16) || (act != CANOPY_ACT_NONE && act != CANOPY_ACT_SILU))
        return CANOPY_ERR_ARG;
    if (B <= 0 || T <= 0 || C <= 0 || K < 2) return CANOPY_ERR_ARG;
    if (T > kMaxT || K > 8 || C % 4 != 0) return CANOPY_ERR_UNSUPPORTED;
    return cuda_status(launch_tree_conv(x, dtype == CANOPY_BF16, conv_state, weight, bias, parent, T, B, C, K,
                                        act == CANOPY_ACT_SILU, y, err, static_cast<cudaStream_t>(stream)));
}

canopy_status canopy_conv_commit(const int32_t* accepted, const void* x, canopy_dtype dtype, const int32_t* parent,
                                 const float* conv_state, float* conv_state_new, int T, int B, int C, int K,
                                 int32_t* err, void* stream) {
    if (!aligned16(accepted) || !aligned16(x) || !aligned16(parent) || !aligned16(conv_state) ||
        !aligned16(conv_state_new) || (err && (reinterpret_cast<uintptr_t>(err) & 3u)))
        return CANOPY_ERR_ARG;
    if (dtype != CANOPY_F32 && dtype != CANOPY_BF16) return CANOPY_ERR_ARG;
    if (B <= 0 || T <= 0 || C <= 0 || K < 2) return CANOPY_ERR_ARG;
    if (T > kMaxT || K > 8 || C % 4 != 0) return CANOPY_ERR_UNSUPPORTED;
    return cuda_status(launch_conv_commit(accepted, x, dtype == CANOPY_BF16, parent, conv_state, conv_state_new, T,
                                          B, C, K, err, static_cast<cudaStream_t>(stream)));
}

canopy_status canopy_read_device_error(void* workspace, int32_t* err_out, void* stream) {
    if (!aligned16(workspace) || !err_out) return CANOPY_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t* dev = static_cast<int32_t*>(workspace);  // the error word is the workspace's first word
    int32_t host = 0;
    if (cudaMemcpyAsync(&host, dev, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return CANOPY_ERR_CUDA;
    if (cudaMemsetAsync(dev, 0, sizeof(int32_t), st) != cudaSuccess) return CANOPY_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return CANOPY_ERR_CUDA;
    *err_out = host;
    return CANOPY_OK;
}

const char* canopy_status_string(canopy_status s) {
    switch (s) {
        case CANOPY_OK: return "ok";
        case CANOPY_ERR_ARG: return "invalid argument";
        case CANOPY_ERR_TREE: return "invalid tree";
        case CANOPY_ERR_UNSUPPORTED: return "unsupported size or combination";
        case CANOPY_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}

int canopy_version(void) { return (0 << 16) | 1; }

}  // extern "C"
