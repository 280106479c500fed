// pkv_decode_noalloc: decode attention for callers that cannot allocate
// device memory.
//
// pkv_decode needs a scratch workspace (per-piece softmax states for the
// split-K merge) that the caller allocates.  Some callers cannot: a plugin
// running inside a host runtime that owns all device memory and hands it only
// the input and output buffers, or a service with a fixed device-memory budget
// that must not grow after start-up.  This entry point uses a scratch array
// that lives in the library itself instead, so it calls no cudaMalloc,
// cudaFree or other allocating routine.
//
// The array is file-scope device memory of a fixed size: every GPU that loads
// the library holds it until the process exits.  Its device address is looked
// up once per device, on that device's first call (with the device current),
// so make that first call before any stream capture.  The cached address
// belongs to the device's current context: it does not survive a
// cudaDeviceReset (or any teardown of the primary context), after which this
// entry point must not be called again in the same process.
//
// All calls share the array and it keeps the last call's contents.  Nothing
// in it needs to start at any particular value: the split-K kernel writes the
// chunk plan and every piece state before the combine reads them, and where
// the combine loads the state of a piece slot that no warp wrote this call
// (its batched loads run ahead of the ownership test), it discards the value
// unused.  Calls that overlap on the GPU (two streams, two host threads) race
// on the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kMaxDevicesNoalloc = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_DECODE_NOALLOC_SCRATCH_BYTES];

void* g_scratch_ptr[kMaxDevicesNoalloc] = {};
std::mutex g_scratch_mu;

// Device address of this device's scratch array, or nullptr on failure.
void* scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNoalloc) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_decode_noalloc(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t batch, int32_t max_context_len,
                                         int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, int32_t num_blocks, float softmax_scale,
                                         pkv_bf16* out, pkv_stream_t stream) {
    if (batch < 0) return PKV_ERR_INVALID_ARG;
    const size_t need = pkv_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim);
    if (need > PKV_DECODE_NOALLOC_SCRATCH_BYTES) return PKV_ERR_UNSUPPORTED;   // batch too large for the array
    void* scratch = pkv::scratch_for_current_device();
    if (scratch == nullptr) return PKV_ERR_CUDA;
    return pkv_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, batch, max_context_len,
                      num_heads, num_kv_heads, head_dim, block_size, num_blocks, softmax_scale, out, scratch,
                      PKV_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
