// mla_sparse_decode_noalloc: the sparse decode for callers that cannot
// allocate device memory at the call site.
//
// mla_sparse_decode needs a caller-provided workspace whenever it splits a
// token's top-k list across CTAs. Some callers have no way to get one: code
// that runs inside another framework's memory pool without an allocator handle,
// or a process that has already reserved all of the device memory it is allowed
// to use. This entry point serves them: its workspace is a fixed array in the
// library's own device memory (kNoAllocScratchBytes below), created when the
// library's device code is loaded on a GPU and held by every GPU that loads the
// library until the process exits. It calls no cudaMalloc, cudaFree or other
// allocating routine.
//
// Rules that follow from the shared array:
//   * every call on a device uses the same array, so calls whose work overlaps
//     on the GPU (different streams, or graphs replayed concurrently) race and
//     give wrong results; serialise them (one stream is enough);
//   * the array keeps whatever the last call left in it. The decode writes every
//     workspace element it later reads, so nothing has to start at zero and no
//     clearing is done;
//   * sizes whose workspace would exceed kNoAllocScratchBytes are rejected with
//     MLA_ENOWORKSPACE before anything is launched;
//   * the first call on each device looks up the array's device address with
//     cudaGetSymbolAddress while that device is current; make that first call
//     before any stream capture.
#include <mutex>

#include "mla_device.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;

// Device-resident scratch. In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (nullptr on error).
void* scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" int mla_sparse_decode_noalloc(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                                         const int32_t* topk_idx, int W, float sm_scale, void* out_bf16,
                                         float* lse, void* stream) {
    // Same split as mla_sparse_decode on this device; reject what does not fit.
    const size_t need = mla_sparse_decode_workspace_bytes(T, H, W);
    if (need > kNoAllocScratchBytes) return MLA_ENOWORKSPACE;
    void* ws = nullptr;
    if (need > 0) {
        ws = scratch_address();
        if (ws == nullptr) return MLA_ECUDA;
    }
    return mla_sparse_decode(q_bf16, T, H, d_qk, kv, topk_idx, W, sm_scale, out_bf16, lse, ws,
                             need > 0 ? kNoAllocScratchBytes : 0, stream);
}
