// libpkv C ABI: argument checks, the per-device error word, tensor-map
// encoding, and dispatch to the kernels of each step.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>
#include <atomic>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kMaxDevices = 64;

// Per-device error word: [0] = PKV_DEVERR_* code, [1] = info.
__device__ int g_error_word[2];

struct DeviceCache {
    int* err = nullptr;
    int sms = 0;
    bool init = false;
};
DeviceCache g_dev[kMaxDevices];
std::mutex g_mu;

DeviceCache* current_cache() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceCache& c = g_dev[dev];
    if (!c.init) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
        c.err = static_cast<int*>(p);
        c.sms = sms;
        c.init = true;
    }
    return &c;
}

std::atomic<bool> g_setup_done[kMaxDevices][kNumSetupKeys];
std::mutex g_setup_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

cudaStream_t as_stream(pkv_stream_t s) { return static_cast<cudaStream_t>(s); }

bool supported_shape(int num_heads, int num_kv_heads, int head_dim, int block_size) {
    return head_dim == kHeadDim && group_log2(num_heads, num_kv_heads) >= 0 && block_size > 0 &&
           block_size % kBlockQuantum == 0;
}

// One thread waits on a barrier that nothing completes, through the bounded wait all the
// kernels use; it gives up after the limit, records the timeout and the kernel returns.
__global__ void wait_check_kernel(int* err) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(b, 0, err, PKV_WAIT_CHECK_INFO);
}

}  // namespace

int* device_error_word() {
    DeviceCache* c = current_cache();
    return c ? c->err : nullptr;
}

int group_log2(int num_heads, int num_kv_heads) {
    if (num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads) return -1;
    const int g = num_heads / num_kv_heads;
    for (int lg = 0; lg <= kMaxLogGroup; ++lg)
        if (g == (1 << lg)) return lg;
    return -1;
}

int sm_count() {
    DeviceCache* c = current_cache();
    return c ? c->sms : 0;
}

bool setup_once(SetupKey key, bool (*setup)()) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::atomic<bool>& done = g_setup_done[dev][key];
    if (done.load(std::memory_order_acquire)) return true;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (done.load(std::memory_order_relaxed)) return true;
    if (!setup()) return false;
    done.store(true, std::memory_order_release);
    return true;
}

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    return fn(map, dtype, rank, base, reinterpret_cast<const cuuint64_t*>(dims),
              reinterpret_cast<const cuuint64_t*>(strides_bytes), reinterpret_cast<const cuuint32_t*>(box),
              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace pkv

using namespace pkv;

extern "C" {

int32_t pkv_abi_version(void) { return 1; }

const char* pkv_status_string(pkv_status status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    }
    return "PKV_ERR_UNKNOWN";
}

pkv_status pkv_slot_mapping(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            const int32_t* context_lens, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, int32_t num_seqs, int32_t total_q,
                            int32_t block_size, int32_t num_blocks, int32_t* slot_mapping,
                            pkv_stream_t stream) {
    if (num_seqs < 0 || total_q < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if ((cu_seqlens_k == nullptr) == (context_lens == nullptr)) return PKV_ERR_INVALID_ARG;
    if (cu_seqlens_q == nullptr && total_q != num_seqs) return PKV_ERR_INVALID_ARG;
    if (total_q == 0) return PKV_OK;
    if (block_tables == nullptr || slot_mapping == nullptr) return PKV_ERR_INVALID_ARG;
    int* err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    const cudaError_t e = launch_slot_mapping(cu_seqlens_q, cu_seqlens_k, context_lens, block_tables,
                                              max_blocks_per_seq, num_seqs, total_q, block_size, num_blocks,
                                              slot_mapping, err, as_stream(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_store_kvcache(const pkv_bf16* k, const pkv_bf16* v, int64_t n_tokens,
                             int64_t k_token_stride, int64_t v_token_stride,
                             const int32_t* slot_mapping, pkv_bf16* k_cache, pkv_bf16* v_cache,
                             int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                             int32_t head_dim, pkv_stream_t stream) {
    if (n_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (k_token_stride < row || v_token_stride < row) return PKV_ERR_INVALID_ARG;
    if (n_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    // 16-byte vector path: rows and their starts must be 16-byte aligned
    if (row % 8 || k_token_stride % 8 || v_token_stride % 8) return PKV_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(k_cache) |
         reinterpret_cast<uintptr_t>(v_cache)) & 15)
        return PKV_ERR_UNSUPPORTED;
    if (n_tokens > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    int* err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    const cudaError_t e = launch_store_kvcache(k, v, n_tokens, k_token_stride, v_token_stride, slot_mapping,
                                               k_cache, v_cache, static_cast<int64_t>(num_blocks) * block_size,
                                               static_cast<int>(row), err, as_stream(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_rope_store_kvcache(const pkv_bf16* q, int64_t q_token_stride, pkv_bf16* q_out,
                                  int64_t q_out_token_stride, const pkv_bf16* k, int64_t k_token_stride,
                                  const pkv_bf16* v, int64_t v_token_stride, const int32_t* positions,
                                  int64_t n_tokens, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, double rope_base, const int32_t* slot_mapping,
                                  pkv_bf16* k_cache, pkv_bf16* v_cache, int32_t num_blocks,
                                  int32_t block_size, pkv_stream_t stream) {
    if (n_tokens < 0 || num_heads < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 ||
        block_size <= 0 || !(rope_base > 0.0) || rope_base == INFINITY)
        return PKV_ERR_INVALID_ARG;
    if ((q == nullptr) != (q_out == nullptr) || (q != nullptr && num_heads == 0)) return PKV_ERR_INVALID_ARG;
    if (head_dim % 16 || head_dim > 2 * kMaxRopePairs) return PKV_ERR_UNSUPPORTED;
    const int64_t kv_row = static_cast<int64_t>(num_kv_heads) * head_dim;
    const int64_t q_row = static_cast<int64_t>(num_heads) * head_dim;
    if (k_token_stride < kv_row || v_token_stride < kv_row) return PKV_ERR_INVALID_ARG;
    if (q && (q_token_stride < q_row || q_out_token_stride < q_row)) return PKV_ERR_INVALID_ARG;
    if (q && q == q_out && q_token_stride != q_out_token_stride) return PKV_ERR_INVALID_ARG;
    if (n_tokens == 0) return PKV_OK;
    if (!k || !v || !positions || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (k_token_stride % 8 || v_token_stride % 8 || (q && (q_token_stride % 8 || q_out_token_stride % 8)))
        return PKV_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(q_out) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(k_cache) |
         reinterpret_cast<uintptr_t>(v_cache)) & 15)
        return PKV_ERR_UNSUPPORTED;
    if (n_tokens > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    RopeStoreArgs a{};
    a.q = q;
    a.q_out = q_out;
    a.k = k;
    a.v = v;
    a.positions = positions;
    a.slots = slot_mapping;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.q_stride = q_token_stride;
    a.q_out_stride = q_out_token_stride;
    a.k_stride = k_token_stride;
    a.v_stride = v_token_stride;
    a.num_slots = static_cast<int64_t>(num_blocks) * block_size;
    a.kv_row = kv_row;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    // pair i advances base^(-2i/d) radians per position: store the fraction of a
    // turn in 64-bit fixed point (whole turns change no angle)
    for (int i = 0; i < head_dim / 2; ++i) {
        const double t = pow(rope_base, -2.0 * i / head_dim) / 6.283185307179586;
        a.turns[i] = static_cast<uint64_t>(ldexp(t - floor(t), 64));   // t - floor(t) < 1: in range
    }
    if (rope_store_threads(a) == 0) return PKV_ERR_UNSUPPORTED;
    int* err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    return launch_rope_store(a, n_tokens, err, as_stream(stream)) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t pkv_prefill_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_seqlen_q) {
    if (num_seqs < 0 || max_seqlen_q < 0 || !supported_shape(num_heads, num_kv_heads, head_dim, kBlockQuantum))
        return 0;
    return prefill_workspace_bytes(num_seqs, max_seqlen_q, group_log2(num_heads, num_kv_heads));
}

namespace {

// Host checks and argument packing shared by the prefill entry points; q, k_cache,
// v_cache and out are only checked when the call attends (not for a plan).
pkv_status prefill_call(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* block_tables,
                        int32_t max_blocks_per_seq, int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                        int32_t max_seqlen_k, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int32_t num_blocks, float softmax_scale, pkv_bf16* out,
                        void* workspace, size_t workspace_bytes, pkv_stream_t stream, pkv::PrefillMode mode) {
    const bool attends = mode != pkv::kPrefillPlanOnly;
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID_ARG;
    if (attends && (num_blocks <= 0 || !(softmax_scale > 0.f) || softmax_scale == INFINITY))
        return PKV_ERR_INVALID_ARG;
    if (!supported_shape(num_heads, num_kv_heads, head_dim, block_size)) return PKV_ERR_UNSUPPORTED;
    if (max_seqlen_q > max_seqlen_k) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return PKV_OK;
    if (!cu_seqlens_q || !cu_seqlens_k) return PKV_ERR_INVALID_ARG;
    if (attends) {
        if (!q || !k_cache || !v_cache || !block_tables || !out) return PKV_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
             reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) & 15)
            return PKV_ERR_UNSUPPORTED;
    }
    if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    int* err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    PrefillArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.block_tables = block_tables;
    a.out = out;
    a.max_blocks = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.total_q = total_q;
    a.max_seqlen_q = max_seqlen_q;
    a.max_seqlen_k = max_seqlen_k;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.softmax_scale = softmax_scale;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launch_prefill(a, err, as_stream(stream), mode);
}

}  // namespace

pkv_status pkv_prefill_varlen(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                              const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                              int32_t max_seqlen_k, int32_t num_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, int32_t num_blocks,
                              float softmax_scale, pkv_bf16* out, void* workspace,
                              size_t workspace_bytes, pkv_stream_t stream) {
    return prefill_call(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, max_blocks_per_seq,
                        num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_dim,
                        block_size, num_blocks, softmax_scale, out, workspace, workspace_bytes, stream,
                        pkv::kPrefillPlanAndRun);
}

pkv_status pkv_prefill_plan(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int32_t max_blocks_per_seq, int32_t num_seqs, int32_t total_q,
                            int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size, void* workspace,
                            size_t workspace_bytes, pkv_stream_t stream) {
    return prefill_call(nullptr, nullptr, nullptr, cu_seqlens_q, cu_seqlens_k, nullptr, max_blocks_per_seq,
                        num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_dim,
                        block_size, 0, 0.f, nullptr, workspace, workspace_bytes, stream, pkv::kPrefillPlanOnly);
}

pkv_status pkv_prefill_varlen_planned(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                                      int32_t max_seqlen_k, int32_t num_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                      float softmax_scale, pkv_bf16* out, void* workspace,
                                      size_t workspace_bytes, pkv_stream_t stream) {
    return prefill_call(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, max_blocks_per_seq,
                        num_seqs, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads, head_dim,
                        block_size, num_blocks, softmax_scale, out, workspace, workspace_bytes, stream,
                        pkv::kPrefillRunOnly);
}

size_t pkv_decode_workspace_size(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                 int32_t head_dim) {
    if (batch < 0 || !supported_shape(num_heads, num_kv_heads, head_dim, kBlockQuantum)) return 0;
    const int W = decode_total_warps();
    if (W <= 0) return 0;
    return decode_workspace_bytes(batch, num_kv_heads, group_log2(num_heads, num_kv_heads), W);
}

pkv_status pkv_decode(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                      const int32_t* context_lens, int32_t batch, int32_t max_context_len,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t num_blocks, float softmax_scale,
                      pkv_bf16* out, void* workspace, size_t workspace_bytes,
                      pkv_stream_t stream) {
    (void)max_context_len;
    if (batch < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_context_len < 0 ||
        !(softmax_scale > 0.f) || softmax_scale == INFINITY)
        return PKV_ERR_INVALID_ARG;
    if (!supported_shape(num_heads, num_kv_heads, head_dim, block_size)) return PKV_ERR_UNSUPPORTED;
    if (batch == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
         reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) & 15)
        return PKV_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_WORKSPACE;
    int* err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    DecodeArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = out;
    a.max_blocks = max_blocks_per_seq;
    a.batch = batch;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.softmax_scale = softmax_scale;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return launch_decode(a, err, as_stream(stream));
}

pkv_status pkv_decode_append(const pkv_bf16* q, const pkv_bf16* k_new, const pkv_bf16* v_new,
                             pkv_bf16* k_cache, pkv_bf16* v_cache, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                             int32_t max_context_len, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t num_blocks, float softmax_scale, pkv_bf16* out,
                             int32_t* slot_mapping, void* workspace, size_t workspace_bytes,
                             pkv_stream_t stream) {
    if (batch < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_context_len < 0 ||
        !(softmax_scale > 0.f) || softmax_scale == INFINITY)
        return PKV_ERR_INVALID_ARG;
    if (!supported_shape(num_heads, num_kv_heads, head_dim, block_size)) return PKV_ERR_UNSUPPORTED;
    if (batch == 0) return PKV_OK;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
         reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) &
        15)
        return PKV_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_WORKSPACE;
    int* err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    DecodeArgs a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = out;
    a.max_blocks = max_blocks_per_seq;
    a.batch = batch;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.softmax_scale = softmax_scale;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.k_new = k_new;
    a.v_new = v_new;
    a.slot_out = slot_mapping;
    return launch_decode(a, err, as_stream(stream));
}

pkv_status pkv_sample(const float* logits, int32_t batch, int32_t vocab, int64_t row_stride,
                      const float* temperatures, uint64_t seed, uint64_t offset, int64_t* out_ids,
                      pkv_stream_t stream) {
    if (batch < 0 || vocab <= 0 || row_stride < vocab) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!logits || !temperatures || !out_ids) return PKV_ERR_INVALID_ARG;
    if (batch > 65535) return PKV_ERR_UNSUPPORTED;
    int* err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    const cudaError_t e = launch_sample(logits, batch, vocab, row_stride, temperatures, seed, offset, nullptr,
                                        out_ids, err, as_stream(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_sample_dev(const float* logits, int32_t batch, int32_t vocab, int64_t row_stride,
                          const float* temperatures, const uint64_t* seed_offset, int64_t* out_ids,
                          pkv_stream_t stream) {
    if (batch < 0 || vocab <= 0 || row_stride < vocab) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!logits || !temperatures || !out_ids || !seed_offset) return PKV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(seed_offset) & 7) return PKV_ERR_INVALID_ARG;
    if (batch > 65535) return PKV_ERR_UNSUPPORTED;
    int* err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    const cudaError_t e = launch_sample(logits, batch, vocab, row_stride, temperatures, 0, 0, seed_offset, out_ids,
                                        err, as_stream(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_check_wait_timeout(pkv_stream_t stream) {
    int* err = device_error_word();
    if (!err) return PKV_ERR_CUDA;
    wait_check_kernel<<<1, 32, 0, as_stream(stream)>>>(err);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_get_device_error(int32_t* code, int32_t* info, int32_t clear) {
    if (!code || !info) return PKV_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
    int h[2] = {0, 0};
    if (cudaMemcpyFromSymbol(h, g_error_word, sizeof(h)) != cudaSuccess) return PKV_ERR_CUDA;
    *code = h[0];
    *info = h[1];
    if (clear) {
        const int z[2] = {0, 0};
        if (cudaMemcpyToSymbol(g_error_word, z, sizeof(z)) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // extern "C"
