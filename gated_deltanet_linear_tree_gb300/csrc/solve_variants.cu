// Solve variants of the tree verify beside the blocked substitution: the
// finite Neumann series, the squaring form and the split design.
//
// canopy page (projects.dotslasha.me/p/canopy.md), "The tree closed form":
// G is nilpotent (G^(d+1) = 0 for a tree of depth d), so
//     (I + G)^-1 = sum_{m=0..d} (-G)^m                      (Neumann series)
//                = (I - G)(I + G^2)(I + G^4) ... (I + G^(2^(k-1))),
// with k = ceil(log2(d + 1)) factors (the squaring form); and "Design
// decisions" (the split alternative: (I + G)^-1 built once per (stream,
// value head) in global memory, then applied per value tile).
//
// All three start from the tensor-core Gram's scratch (gram_tc.cu): G and C
// as [B][H][T][T] (64 x 64 tiles on and below the diagonal, zero off the
// paths), gamma X_Q and R as [B][T][H][dv]; like the blocked substitution
// they write U = (I + G)^-1 R to the workspace (the commit reads it) and
//     o = scale (gamma X_Q + C U).
// Each runs on tcgen05 tensor cores with the lower-triangular tile product of
// tc_tiles.cuh: neumann_tc.cu (T > 64; the one-block Neumann series is part
// of verify_tc.cu), squaring_tc.cu and split_tc.cu.  The squaring form and
// the split design overwrite the G and C scratch, which nothing reads after
// the verify.
#include "common.cuh"

namespace canopy {

cudaError_t launch_neumann_tc(int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st);
cudaError_t launch_squaring_tc(int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st);
cudaError_t launch_split_tc(int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws, cudaStream_t st);

// variant: 1 Neumann series (T > 64), 2 squaring form, 3 split design
// (dk = dv = 128).  The Gram scratch must be in place (launch_gram_tc).
cudaError_t launch_solve_variant(int variant, int T, int B, int H, void* o, int o_bf16, float scale, const Ws& ws,
                                 cudaStream_t st) {
    if (T < 1 || T > kMaxT) return cudaErrorInvalidValue;
    if (variant == 1) return launch_neumann_tc(T, B, H, o, o_bf16, scale, ws, st);
    if (variant == 2) return launch_squaring_tc(T, B, H, o, o_bf16, scale, ws, st);
    if (variant == 3) return launch_split_tc(T, B, H, o, o_bf16, scale, ws, st);
    return cudaErrorInvalidValue;
}

}  // namespace canopy
