// Serial replay with its snapshot scratch in a fixed device array, for
// callers that cannot allocate device memory.
//
// Some hosts own all device memory through their own allocator (an
// inference server's memory pool, a framework arena with a fixed budget) and
// do not let a library make side allocations; some latency-critical loops
// cannot afford cudaMalloc, which may synchronise the device.  Such callers
// cannot provide the snapshot buffer that canopy_serial_replay needs.  This
// entry point uses a file-scope device array instead: the library reserves
// it on every GPU that loads the module, and keeps it until the process
// exits.  The kernel is the same serial replay kernel as canopy_serial_replay.
#include <mutex>

#include "common.cuh"

namespace canopy {
cudaError_t launch_serial(const void* q, const void* k, const void* v, int in_bf16, const float* g,
                          const float* beta, const float* S0, const int32_t* parent, int T, int B, int H, int HK,
                          int d, void* o, int o_bf16, float scale, float* snap, int32_t* err, cudaStream_t st);
}  // namespace canopy

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB of per-node snapshots

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol; kernels receive the address that cudaGetSymbolAddress
// returns for the current device.
static __device__ __align__(256) unsigned char g_snapshot_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Once per device, with that device current: look up the array's address.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_snapshot_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite(float x) { return x == x && x - x == 0.f; }

}  // namespace

extern "C" {

canopy_status canopy_serial_replay_static(const void* q, const void* k, const void* v, canopy_dtype in_dtype,
                                          const float* g, const float* beta, const float* S0,
                                          const int32_t* parent, int T, int B, int H, int HV, int dk, int dv,
                                          float scale, void* o, canopy_dtype o_dtype, int32_t* err, void* stream) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) || !aligned16(S0) ||
        !aligned16(parent) || !aligned16(o) || (err && (reinterpret_cast<uintptr_t>(err) & 3u)))
        return CANOPY_ERR_ARG;
    if ((in_dtype != CANOPY_F32 && in_dtype != CANOPY_BF16) || (o_dtype != CANOPY_F32 && o_dtype != CANOPY_BF16) ||
        !finite(scale))
        return CANOPY_ERR_ARG;
    if (B <= 0 || H <= 0 || T <= 0 || HV < H || HV % H != 0) return CANOPY_ERR_ARG;
    if (T > canopy::kMaxT || dk != dv || (dk != 128 && dk != 32)) return CANOPY_ERR_UNSUPPORTED;
    const size_t need = size_t(B) * T * HV * dv * dk * 4;
    if (need > kScratchBytes - 256) return CANOPY_ERR_UNSUPPORTED;  // the last 256 bytes hold a spare error word
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return CANOPY_ERR_CUDA;
    // A null err goes to a word inside the scratch, past the snapshots used.
    int32_t* err_word = err ? err : reinterpret_cast<int32_t*>(static_cast<char*>(scratch) + kScratchBytes - 256);
    cudaError_t e = canopy::launch_serial(q, k, v, in_dtype == CANOPY_BF16, g, beta, S0, parent, T, B, HV, H, dk, o,
                                          o_dtype == CANOPY_BF16, scale, static_cast<float*>(scratch), err_word,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CANOPY_OK : CANOPY_ERR_CUDA;
}

}  // extern "C"
