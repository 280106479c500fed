// a1 slot mapping and a2 KV scatter.
//
// Slot rule: visual atlas (diomchen.github.io/reference/visual-atlas.html),
// figure "T=5, block_size=2, block_table=[3,0,4]".  Scatter: nano-vLLM offline
// explainer, accuracy & scope box ("input tokens write KV, then sample").
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// One thread per new token.  Sequence of packed token t: the s with
// cu_q[s] <= t < cu_q[s+1] (binary search), or s = t when cu_q is null.
__global__ void slot_mapping_kernel(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k,
                                    const int32_t* __restrict__ ctx,
                                    const int32_t* __restrict__ block_tables, int max_blocks,
                                    int num_seqs, int total_q, int block_size, int num_blocks,
                                    int32_t* __restrict__ slots, int* err) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= total_q) return;
    int s, q_start, q_len;
    if (cu_q == nullptr) {
        s = t;
        q_start = t;
        q_len = 1;
    } else {
        int lo = 0, hi = num_seqs;               // find last s with cu_q[s] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(cu_q + mid) <= t) lo = mid; else hi = mid;
        }
        s = lo;
        q_start = __ldg(cu_q + s);
        q_len = __ldg(cu_q + s + 1) - q_start;
    }
    const int k_len = (cu_k != nullptr) ? __ldg(cu_k + s + 1) - __ldg(cu_k + s) : __ldg(ctx + s);
    if (q_len > k_len || q_len < 0) {
        record_error(err, PKV_DEVERR_SEQLENS, s);
        slots[t] = -1;
        return;
    }
    const int pos = k_len - q_len + (t - q_start);
    const int logical = pos / block_size;
    if (logical >= max_blocks) {
        record_error(err, PKV_DEVERR_BLOCK_TABLE, t);
        slots[t] = -1;
        return;
    }
    const int phys = __ldg(block_tables + static_cast<int64_t>(s) * max_blocks + logical);
    if (phys < 0 || phys >= num_blocks) {
        record_error(err, PKV_DEVERR_BLOCK_ID, t);
        slots[t] = -1;
        return;
    }
    slots[t] = phys * block_size + (pos - logical * block_size);
}

// One CTA per token row; each thread moves 16-byte vectors of K then V.
// Loads go through the non-coherent path and are marked streaming; the
// destination rows are scattered 2 KiB rows of the pool.
__global__ void __launch_bounds__(128) store_kvcache_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t k_stride,
    int64_t v_stride, const int32_t* __restrict__ slots, uint16_t* __restrict__ k_cache,
    uint16_t* __restrict__ v_cache, int64_t num_slots, int row_vecs, int* err) {
    const int64_t i = blockIdx.x;
    const int slot = __ldg(slots + i);
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0) record_error(err, PKV_DEVERR_SLOT, static_cast<int>(i));
        return;
    }
    const uint4* ks = reinterpret_cast<const uint4*>(k + i * k_stride);
    const uint4* vs = reinterpret_cast<const uint4*>(v + i * v_stride);
    uint4* kd = reinterpret_cast<uint4*>(k_cache) + static_cast<int64_t>(slot) * row_vecs;
    uint4* vd = reinterpret_cast<uint4*>(v_cache) + static_cast<int64_t>(slot) * row_vecs;
    for (int j = threadIdx.x; j < row_vecs; j += blockDim.x) {
        const uint4 a = __ldcs(ks + j);
        const uint4 b = __ldcs(vs + j);
        kd[j] = a;
        vd[j] = b;
    }
}

}  // namespace

cudaError_t launch_slot_mapping(const int32_t* cu_q, const int32_t* cu_k, const int32_t* ctx,
                                const int32_t* block_tables, int max_blocks, int num_seqs,
                                int total_q, int block_size, int num_blocks, int32_t* slots,
                                int* err, cudaStream_t stream) {
    if (total_q == 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = (total_q + threads - 1) / threads;
    slot_mapping_kernel<<<blocks, threads, 0, stream>>>(cu_q, cu_k, ctx, block_tables, max_blocks,
                                                         num_seqs, total_q, block_size, num_blocks,
                                                         slots, err);
    return cudaGetLastError();
}

cudaError_t launch_store_kvcache(const uint16_t* k, const uint16_t* v, int64_t n_tokens,
                                 int64_t k_stride, int64_t v_stride, const int32_t* slots,
                                 uint16_t* k_cache, uint16_t* v_cache, int64_t num_slots,
                                 int row_elems, int* err, cudaStream_t stream) {
    if (n_tokens == 0) return cudaSuccess;
    const int row_vecs = row_elems / 8;
    store_kvcache_kernel<<<static_cast<unsigned>(n_tokens), 128, 0, stream>>>(
        k, v, k_stride, v_stride, slots, k_cache, v_cache, num_slots, row_vecs, err);
    return cudaGetLastError();
}

}  // namespace pkv
