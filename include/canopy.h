/*
 * canopy: closed-form tree verification for Gated DeltaNet layers on one
 * NVIDIA GB300 (sm_103a).  C ABI of libcanopy.so.
 *
 * The method (canopy page, projects.dotslasha.me/p/canopy.md, "The tree
 * closed form", which states Bole's Theorem 1): a draft tree of T nodes per
 * stream, given as a parent array in any topological order, is verified by
 * one ancestor-masked, decay-weighted unit-lower-triangular solve instead of
 * forking a d_v x d_k state per branch; afterwards only the accepted node's
 * state is rebuilt (commit).  In this library's orientation the state is
 * S[dv][dk] and the rule ("The gated delta rule", TreeWY's form) is
 *     S_i = g_i * S_parent(i) * (I - beta_i k_i k_i^T) + beta_i v_i k_i^T
 *     o_i = S_i (scale * q_i)           (S_parent(0) = S0)
 * with g_i the decay gate alpha_i in (0, 1].  Heads ("Qwen3.5-9B shapes"
 * and "Design decisions", memory layout): q and k have H key heads; v, g,
 * beta, S0, o and the workspace have HV value heads, HV a multiple of H, and
 * value head j reads key head j / (HV / H) (grouped value attention; HV = H
 * is one q/k per head).  scale is the factor on q (1/sqrt(dk) in FLA; 1 for
 * the plain rule).
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers; the caller owns and
 *     allocates every buffer.  The library never allocates, frees or
 *     synchronises inside a compute call; work is enqueued on `stream`
 *     (a cudaStream_t passed as void*, NULL = legacy default stream).
 *   - All arrays are dense, row-major, with the last index fastest:
 *       q, k     [B][T][H][dk]    bf16 or fp32 (in_dtype)
 *       v        [B][T][HV][dv]   bf16 or fp32 (in_dtype)
 *       g, beta  [B][T][HV]       fp32 (g = decay gate alpha, linear space)
 *       S0       [B][HV][dv][dk]  fp32
 *       parent   [B][T]           int32, parent[b][0] = -1, 0 <= parent[b][i] < i
 *       o        [B][T][HV][dv]   fp32 or bf16 (o_dtype)
 *   - Device pointers must be 16-byte aligned (vector and TMA loads).
 *   - Argument errors are detected on the host and returned before anything
 *     is enqueued.  Errors that depend on device data (a malformed tree, a
 *     gate <= 0 or not finite, an accepted node out of range, an internal
 *     wait that timed out) set bits in a sticky device error word inside the
 *     workspace; the outputs of that call are then undefined.  Read and clear
 *     the word with canopy_read_device_error().  No kernel traps or asserts.
 *   - Sizes supported: 1 <= T <= 256, B >= 1, H >= 1, HV a multiple of H
 *     (HV = H where an entry point takes one head count), dk = dv = 128 for every
 *     entry point; dk = dv = 32 additionally for the fp32 (tier A) and serial
 *     paths.  Other values return CANOPY_ERR_UNSUPPORTED.
 */
#ifndef CANOPY_H
#define CANOPY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CANOPY_OK = 0,
    CANOPY_ERR_ARG = 1,          /* null/misaligned pointer, bad enum, B/H/T <= 0   */
    CANOPY_ERR_TREE = 2,         /* reserved for host-side tree checks              */
    CANOPY_ERR_UNSUPPORTED = 3,  /* a size or combination this build does not have  */
    CANOPY_ERR_CUDA = 4          /* a CUDA runtime call failed (launch, copy, ...)  */
} canopy_status;

typedef enum { CANOPY_F32 = 0, CANOPY_BF16 = 1 } canopy_dtype;

/* Solve strategy for (I + diag(beta) A) U = R (canopy page, "Design
 * decisions", solve strategies behind one interface, and "The tree closed
 * form", nilpotency and squaring).  FWDSUB takes every size and dtype; the
 * other three take bf16 q/k/v with dk = dv = 128 only (else
 * CANOPY_ERR_UNSUPPORTED) and never take the path-replay dispatch below.
 * The two series forms (NEUMANN, SQUARING) are accurate while the terms
 * (-G)^m R stay small: on deep paths whose keys are nearly aligned the terms
 * grow before they cancel and fp32 loses them (a 64-node chain of identical
 * keys gives errors of order 1); FWDSUB and SPLIT solve by substitution,
 * whose accuracy does not depend on depth (about 1e-6 in fp32 arithmetic at
 * any depth).  Every strategy multiplies on tcgen05 tensor cores with split
 * bf16 operands (1e-4 to 3e-4 max/rms on the pages' bf16 inputs). */
typedef enum {
    CANOPY_SOLVE_FWDSUB = 0,   /* blocked forward substitution, 64-node blocks            */
    CANOPY_SOLVE_NEUMANN = 1,  /* finite Neumann series, d rounds (Bole's solve)          */
    CANOPY_SOLVE_SQUARING = 2, /* (I - G)(I + G^2)(I + G^4)..., ceil(log2(d + 1)) factors  */
    CANOPY_SOLVE_SPLIT = 3     /* (I + G)^-1 and C (I + G)^-1 once per (stream, value
                                  head) in the workspace, then applied to R by a second
                                  launch (all 128 value columns as one tile)              */
} canopy_solve;

/* Flags of canopy_tree_verify. */
#define CANOPY_VERIFY_INPUTS_READY 0x1u  /* q, k, v, g, beta, parent are not written by the
                                            kernel launched just before this call */
#define CANOPY_VERIFY_STATE_READY 0x2u   /* S0 is not written by the kernel launched just
                                            before this call */
#define CANOPY_VERIFY_CLOSED_FORM 0x4u   /* FWDSUB: never the path replay below the crossover */
#define CANOPY_VERIFY_PATH_REPLAY 0x8u   /* FWDSUB: always the path replay (T <= 8; larger T
                                            returns CANOPY_ERR_UNSUPPORTED) */

/* How a verify call is carried out (canopy_verify_plan). */
typedef enum {
    CANOPY_PLAN_NONE = -1,        /* the call would be refused (an argument error)           */
    CANOPY_PLAN_PATH_REPLAY = 0,  /* each node's root path replayed from S0 (tiny trees)     */
    CANOPY_PLAN_TC_BLOCK = 1,     /* one tensor-core launch, one 64-node block (T <= 64)     */
    CANOPY_PLAN_TC_NEUMANN = 2,   /* the same with the Neumann series                         */
    CANOPY_PLAN_TC_BLOCKED = 3,   /* one tensor-core launch, 64-node blocks in order (T > 64) */
    CANOPY_PLAN_FP32 = 4,         /* tree prep, Gram and level solve in fp32 on CUDA cores   */
    CANOPY_PLAN_VARIANT = 5       /* tree prep, tensor-core Gram, then the solve variant     */
} canopy_plan;

/* Flags of canopy_commit. */
#define CANOPY_COMMIT_STATE_READY 0x1u   /* S0, accepted, k and parent are not written by
                                            the kernel launched just before this call */

/* Bits of the device error word. */
#define CANOPY_DEVERR_TREE     0x1  /* parent[b][0] != -1 or parent[b][i] not in [0,i) */
#define CANOPY_DEVERR_GATE     0x2  /* g <= 0, g or beta not finite                     */
#define CANOPY_DEVERR_ACCEPTED 0x4  /* commit: accepted node not in [-1, T)             */
#define CANOPY_DEVERR_TIMEOUT  0x8  /* an internal bounded wait gave up                 */
#define CANOPY_DEVERR_LENGTH   0x10 /* verify/commit: lengths[b] not in [0, T]           */

/* Size in bytes of the workspace one verify/commit pair needs, for HV value
 * heads.  It holds the pseudo-values U fp32 [B][T][HV][dv], the cumulative
 * log gates l fp32 [B][T][HV] (l_i = sum of log g over path(i)), node depths int32
 * [B][T], the strict-ancestor bitmask uint32 [B][T][ceil(T/32)], the DFS
 * pre-order int32 [B][T], the device error word, and the scratch of the
 * paths beyond one fused launch (the fp32 path, trees of more than 64 nodes
 * and the Neumann, squaring and split solves): G and C as [B][HV][T][T]
 * fp32, gamma X_Q and R as [B][T][HV][dv] fp32.  The squaring and split
 * solves overwrite G and C with G^(2^m), or with (I + G)^-1 and C (I + G)^-1.
 * Returns 0 for unsupported sizes. */
size_t canopy_workspace_bytes(int B, int T, int HV, int dk, int dv);

/* Regions of the workspace that hold results a caller may read (the rest is
 * scratch with no stable contents). */
typedef enum {
    CANOPY_WS_ERR = 0,    /* int32: the sticky device error word (always at offset 0)   */
    CANOPY_WS_L = 1,      /* fp32 [B][T][HV]: l_i, natural log                           */
    CANOPY_WS_DEPTH = 2,  /* int32 [B][T]: |A(i)|                                       */
    CANOPY_WS_MASK = 3,   /* uint32 [B][T][ceil(T/32)]: bit j%32 of word j/32 set iff j
                             is a strict ancestor of i                                   */
    CANOPY_WS_ORDER = 4,  /* int32 [B][T]: DFS pre-order, children in index order
                             (order[b][pos] = node; written by canopy_tree_prep only)    */
    CANOPY_WS_U = 5       /* fp32 [B][T][HV][dv]: the pseudo-values U                    */
} canopy_ws_region;

/* Byte offset of a region inside a workspace of canopy_workspace_bytes(B, T,
 * HV, dk, dv) bytes (every region starts on a 256-byte boundary); (size_t)-1
 * for unsupported sizes or an unknown region.  Host-only, no CUDA call. */
size_t canopy_workspace_offset(int B, int T, int HV, int dk, int dv, canopy_ws_region region);

/* Zero the workspace (including the error word); call once after allocating
 * it.  Enqueued on `stream`. */
canopy_status canopy_workspace_init(void* workspace, size_t bytes, void* stream);

/* Tree preparation (canopy page, "The tree closed form" and "Design
 * decisions", tree order and tiling): validates every parent array and
 * writes depth, the strict-ancestor bitmask, the DFS pre-order and the
 * cumulative log gates l into the workspace.  The verify entry point does the
 * same work inside its own kernels; this call exposes it on its own.
 *   parent device int32 [B][T]; g device fp32 [B][T][HV]. */
canopy_status canopy_tree_prep(const int32_t* parent, const float* g,
                               int T, int B, int HV, void* workspace, void* stream);

/* Closed-form tree verify (canopy page, "The tree closed form"):
 *   A_ij = [j in A(i)] exp(l_i - l_j) k_i.k_j,  C_ij = [j in path(i)] exp(l_i - l_j) q_i.k_j
 *   (I + diag(beta) A) U = diag(beta) (V - diag(gamma) K S0^T),  gamma_i = exp(l_i)
 *   O = diag(gamma) Q S0^T + C U
 * Writes o (device, o_dtype) and, into the workspace, U, l, depth, mask.
 * in_dtype CANOPY_BF16 selects the tensor-core path (tcgen05, bf16 operands,
 * fp32 accumulation); CANOPY_F32 selects the fp32 path.  S0 is read only.
 * With solve = CANOPY_SOLVE_FWDSUB, trees below the measured crossover (one
 * or two nodes; three with B * HV <= 128) are verified by replaying
 * each node's root path from S0 in fp32 instead (same outputs and workspace
 * contents; canopy page, "Design decisions": serial below the crossover).
 * flags: 0, or CANOPY_VERIFY_INPUTS_READY, optionally with
 * CANOPY_VERIFY_STATE_READY.  The tensor-core forward-substitution kernel is
 * launched with programmatic dependent launch and may begin while the kernel
 * launched just before it on `stream` finishes.  With flags = 0 it touches
 * no global memory until that kernel has completed.  With
 * CANOPY_VERIFY_INPUTS_READY the caller asserts that q, k, v, g, beta and
 * parent are not written by that kernel: the call then reads them (and runs
 * tree prep and the triangular solve) while it finishes.  Adding
 * CANOPY_VERIFY_STATE_READY asserts the same of S0 (for instance, the
 * preceding kernel is another layer's verify or commit): S0 is then read
 * early too.  The workspace and o are written only after that kernel has
 * completed, whatever the flags.  CANOPY_VERIFY_STATE_READY without
 * CANOPY_VERIFY_INPUTS_READY has no effect; other bits return
 * CANOPY_ERR_ARG.
 * lengths (canopy page, "Design decisions", memory layout: the parent array
 * plus a per-sequence length for ragged batches): device int32 [B], or NULL
 * when every stream has T nodes.  Stream b's tree is nodes 0 .. lengths[b]-1
 * (0 <= lengths[b] <= T; T stays the stride of every array).  The rows of
 * q, k, v, g, beta and parent past a stream's length do not influence any
 * result, whatever they hold, and the rows of o and of the workspace (U, l,
 * depth, mask) past it are not written.  A length outside [0, T] sets
 * CANOPY_DEVERR_LENGTH and is read as the nearest bound.  The solve variants
 * (NEUMANN, SQUARING, SPLIT) take no lengths: non-NULL returns
 * CANOPY_ERR_UNSUPPORTED. */
canopy_status canopy_tree_verify(const void* q, const void* k, const void* v, canopy_dtype in_dtype,
                                 const float* g, const float* beta, const float* S0,
                                 const int32_t* parent, const int32_t* lengths, int T, int B, int H, int HV,
                                 int dk, int dv, float scale, canopy_solve solve, void* o,
                                 canopy_dtype o_dtype, void* workspace, unsigned flags, void* stream);

/* The plan canopy_tree_verify follows for these sizes, dtype, solve and
 * flags, with lengths given (has_lengths != 0) or not; CANOPY_PLAN_NONE where
 * the call would return an error for them.  The dispatch below the crossover
 * (canopy page, "Design decisions": the serial path below the crossover, the
 * closed form above it) sends trees of one or two nodes, and three-node trees
 * over at most 128 (stream, value head) pairs, to the path replay.
 * Host-only, no CUDA call. */
canopy_plan canopy_verify_plan(int T, int B, int H, int HV, canopy_dtype in_dtype, int dk, int dv,
                               canopy_solve solve, unsigned flags, int has_lengths);

/* Commit (canopy page, "The tree closed form", last line, and "What the
 * commit kernel stores"): for every stream b with accepted node a = accepted[b],
 *   S_new = gamma_a S0 + sum_{j in path(a)} exp(l_a - l_j) u_j k_j^T      (fp32)
 * using U and l that the preceding verify call left in the workspace, and
 * that call's k and parent (path(a) is walked up the parent array, parents
 * sanitised as the verify does).  a = -1 means nothing accepted: S_new = S0.
 * S_new may alias S0 (the update is elementwise in S0).
 * flags: 0 or CANOPY_COMMIT_STATE_READY.  The kernel is launched with
 * programmatic dependent launch; with flags = 0 it touches no global memory
 * until the kernel launched just before it on `stream` has completed.  With
 * CANOPY_COMMIT_STATE_READY the caller asserts that S0, accepted, k and
 * parent are not written by that kernel (a verify call only reads them):
 * the commit then requests its S0 tiles, walks the accepted path and stages
 * its k rows while that kernel finishes; the workspace and S_new are touched
 * only after it has completed.  Other bits return CANOPY_ERR_ARG.
 *   accepted device int32 [B]; S0, S_new device fp32 [B][HV][dv][dk];
 *   k device [B][T][H][dk] in in_dtype; parent device int32 [B][T];
 *   lengths: the verify call's (device int32 [B] or NULL); an accepted node
 *   at or past its stream's length sets CANOPY_DEVERR_ACCEPTED and keeps S0. */
canopy_status canopy_commit(const int32_t* accepted, const float* S0, float* S_new,
                            const void* k, const int32_t* parent, const int32_t* lengths,
                            canopy_dtype in_dtype, int T, int B, int H, int HV, int dk, int dv,
                            const void* workspace, unsigned flags, void* stream);

/* Activation after the short convolution. */
typedef enum { CANOPY_ACT_NONE = 0, CANOPY_ACT_SILU = 1 } canopy_activation;

/* Tree-aware short causal convolution (canopy page, "M7: Benchmarks, the
 * crossover, and the stretch goal": the kernel-4 convolution before each
 * GDN layer follows each node's root path).  Per stream b, node i and
 * channel c, with a_0(i) = i, a_m(i) = parent(a_{m-1}(i)) and depth(i) the
 * number of edges from the root:
 *   y_i[c] = act(bias[c] + sum_{j=0..K-1} w[c][j] X(i, K-1-j)[c]),
 *   X(i, m) = x_{a_m(i)} for m <= depth(i), else
 *             conv_state[c][K-1-(m-depth(i))] (the committed inputs before
 *             the root, [K-2] the newest).
 *   x, y device [B][T][C] in dtype (bf16 or fp32; fp32 arithmetic);
 *   conv_state device fp32 [B][C][K-1]; weight device fp32 [C][K]; bias
 *   device fp32 [C] or NULL; parent device int32 [B][T] (sanitised as the
 *   verify sanitises it; a bad tree sets CANOPY_DEVERR_TREE in *err).
 *   2 <= K <= 8; C a multiple of 4; err an optional device int32 (OR-ed).
 * Enqueued on `stream`; no allocation. */
canopy_status canopy_tree_conv(const void* x, canopy_dtype dtype, const float* conv_state, const float* weight,
                               const float* bias, const int32_t* parent, int T, int B, int C, int K,
                               canopy_activation act, void* y, int32_t* err, void* stream);

/* Convolution-state commit (same passage: commit updates the convolution
 * state with the accepted tokens): for accepted node a = accepted[b] the new
 * state is the last K-1 inputs of (conv_state ++ x over path(a), root
 * first); a = -1 keeps the state, a outside [-1, T) sets
 * CANOPY_DEVERR_ACCEPTED in *err and keeps it.  conv_state_new may alias
 * conv_state.  Shapes as in canopy_tree_conv; accepted device int32 [B]. */
canopy_status canopy_conv_commit(const int32_t* accepted, const void* x, canopy_dtype dtype, const int32_t* parent,
                                 const float* conv_state, float* conv_state_new, int T, int B, int C, int K,
                                 int32_t* err, void* stream);

/* Bytes of the per-node snapshot buffer of the serial replay for HV value
 * heads: fp32 [B][T][HV][dv][dk]. */
size_t canopy_snapshot_bytes(int B, int T, int HV, int dk, int dv);

/* Serial parent-pointer replay, the crossover opponent (canopy page,
 * "Design decisions", serial baseline: SGLang's snapshot path).  For each
 * node in index order it takes the parent's state (S0 for the root) from the
 * snapshot buffer, applies one step of the rule in fp32, writes the node's
 * snapshot when a later node other than i+1 will read it, and writes o_i.
 * Same inputs and output as canopy_tree_verify; snapshot is device memory of
 * canopy_snapshot_bytes(); workspace receives only the error word. */
canopy_status canopy_serial_replay(const void* q, const void* k, const void* v, canopy_dtype in_dtype,
                                   const float* g, const float* beta, const float* S0,
                                   const int32_t* parent, int T, int B, int H, int HV, int dk, int dv,
                                   float scale, void* o, canopy_dtype o_dtype, void* snapshot,
                                   void* workspace, void* stream);

/* Serial replay for callers that cannot allocate device memory.  The paper
 * has no counterpart: this is a deployment variant of canopy_serial_replay.
 * Hosts that own every device allocation through their own pool, or loops
 * that cannot pay for cudaMalloc's device synchronisation, cannot hand the
 * library a snapshot buffer; this call keeps its per-node snapshots in a
 * fixed 32 MiB device array inside the library instead, reserved on every
 * GPU that loads the library and held until the process exits.
 *   - Same inputs and output o as canopy_serial_replay; no workspace and no
 *     snapshot argument.  err is an optional device int32 (may be NULL):
 *     device-side input errors (CANOPY_DEVERR_*) are OR-ed into it, so zero
 *     it before the call if you read it afterwards.
 *   - Limit: B*T*HV*dk*dv*4 <= 33,554,176 bytes (32 MiB less 256 bytes), e.g.
 *     B=1, T=31, HV=16 at dk=dv=128; larger calls return
 *     CANOPY_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on a device looks up the array's address there
 *     (cudaGetSymbolAddress, with that device current) and keeps it for the
 *     life of the process; make that first call before any stream capture.
 *     The kept address belongs to the device's context at that time: after a
 *     cudaDeviceReset (or any teardown of that context) do not call this
 *     entry point again in the same process.
 *   - All calls share the one array, which keeps the last call's contents;
 *     nothing in it needs to start at zero (every snapshot is written before
 *     it is read), but calls that overlap on the GPU race with each other.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine. */
canopy_status canopy_serial_replay_static(const void* q, const void* k, const void* v, canopy_dtype in_dtype,
                                          const float* g, const float* beta, const float* S0,
                                          const int32_t* parent, int T, int B, int H, int HV, int dk,
                                          int dv, float scale, void* o, canopy_dtype o_dtype, int32_t* err,
                                          void* stream);

/* Synchronise `stream`, copy the device error word to *err_out and clear it.
 * Returns CANOPY_ERR_CUDA if the stream reported an error. */
canopy_status canopy_read_device_error(void* workspace, int32_t* err_out, void* stream);

/* Human-readable name of a status. */
const char* canopy_status_string(canopy_status s);

/* Version of this library as (major << 16) | minor. */
int canopy_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CANOPY_H */
