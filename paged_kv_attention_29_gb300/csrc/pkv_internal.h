// Host-side declarations shared by the libpkv translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

constexpr int kHeadDim = 128;
constexpr int kMaxLogGroup = 3;      // query heads per KV head: 1, 2, 4 or 8
constexpr int kBlockQuantum = 256;   // block_size must be a multiple of this

// log2(num_heads / num_kv_heads) when that ratio is 1, 2, 4 or 8; otherwise -1.
int group_log2(int num_heads, int num_kv_heads);

// Device address of the current device's error word (int[2]); nullptr on failure.
int* device_error_word();

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// One-time set-up of kernel attributes, per device.  Runs `setup` with the
// current device once (thread-safe; a failed set-up is retried on the next
// call) and returns whether the set-up for `key` has succeeded on this device.
enum SetupKey { kSetupDecode = 0, kSetupPrefill, kSetupRopeStore, kNumSetupKeys };
bool setup_once(SetupKey key, bool (*setup)());

// cuTensorMapEncodeTiled through the runtime's driver entry point.
CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle);

// ---- a1 / a2 --------------------------------------------------------------
cudaError_t launch_slot_mapping(const int32_t* cu_q, const int32_t* cu_k, const int32_t* ctx,
                                const int32_t* block_tables, int max_blocks, int num_seqs,
                                int total_q, int block_size, int num_blocks, int32_t* slots,
                                int* err, cudaStream_t stream);

cudaError_t launch_store_kvcache(const uint16_t* k, const uint16_t* v, int64_t n_tokens,
                                 int64_t k_stride, int64_t v_stride, const int32_t* slots,
                                 uint16_t* k_cache, uint16_t* v_cache, int64_t num_slots,
                                 int row_elems, int* err, cudaStream_t stream);

// ---- f2: RoPE fused into the KV write -------------------------------------------
constexpr int kMaxRopePairs = 128;   // head_dim <= 256

struct RopeStoreArgs {
    const uint16_t* q;        // nullptr: rotate and store K only
    uint16_t* q_out;
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* positions;
    const int32_t* slots;
    uint16_t* k_cache;
    uint16_t* v_cache;
    int64_t q_stride, q_out_stride, k_stride, v_stride;   // elements between tokens
    int64_t num_slots;
    int64_t kv_row;            // num_kv_heads * head_dim
    int num_heads, num_kv_heads, head_dim;
    uint64_t turns[kMaxRopePairs];    // 2^64 * frac(base^(-2i/d) / (2 pi)), i < d/2
};

// Threads one CTA needs (one per work item of a token); 0 if above 1024.
int rope_store_threads(const RopeStoreArgs& a);
cudaError_t launch_rope_store(const RopeStoreArgs& a, int64_t n_tokens, int* err, cudaStream_t stream);

// ---- a4 ---------------------------------------------------------------------
struct DecodeArgs {
    const uint16_t* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    uint16_t* out;
    int max_blocks;
    int batch;
    int num_heads;
    int num_kv_heads;
    int block_size;
    int num_blocks;
    float softmax_scale;
    void* workspace;
    size_t workspace_bytes;
    const uint16_t* k_new = nullptr;   // fused KV write (pkv_decode_append); nullptr: none
    const uint16_t* v_new = nullptr;
    int32_t* slot_out = nullptr;
};

int decode_total_warps();                                  // warps the decode grid runs
size_t decode_workspace_bytes(int batch, int num_kv_heads, int log_group, int total_warps);
pkv_status launch_decode(const DecodeArgs& a, int* err, cudaStream_t stream);

// ---- a3 ---------------------------------------------------------------------
struct PrefillArgs {
    const uint16_t* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* cu_q;
    const int32_t* cu_k;
    const int32_t* block_tables;
    uint16_t* out;
    int max_blocks;
    int num_seqs;
    int total_q;
    int max_seqlen_q;
    int max_seqlen_k;
    int num_heads;
    int num_kv_heads;
    int block_size;
    int num_blocks;
    float softmax_scale;
    void* workspace;
    size_t workspace_bytes;
};

// log_group = log2(num_heads / num_kv_heads)
size_t prefill_workspace_bytes(int num_seqs, int max_seqlen_q, int log_group);
// kPrefillPlanAndRun: plan the work list into the workspace, then attend;
// kPrefillPlanOnly: the plan alone; kPrefillRunOnly: attend on the plan already
// in the workspace (made for the same lengths, bounds and group size).
enum PrefillMode { kPrefillPlanAndRun, kPrefillPlanOnly, kPrefillRunOnly };
pkv_status launch_prefill(const PrefillArgs& a, int* err, cudaStream_t stream, PrefillMode mode);

// ---- a5 ---------------------------------------------------------------------
cudaError_t launch_sample(const float* logits, int batch, int vocab, int64_t row_stride,
                          const float* temperatures, uint64_t seed, uint64_t offset,
                          const uint64_t* seed_offset, int64_t* out_ids, int* err, cudaStream_t stream);

}  // namespace pkv
