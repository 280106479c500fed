// f2: rotary position embedding fused into the KV write.
//
// Visual atlas (diomchen.github.io/reference/visual-atlas.html), fig. 19: each
// head splits into d/2 two-dimensional pairs, pair i turned by an angle that
// grows with the position at its own frequency; the engine rotates Q and K and
// leaves V as it is.  The rotated K row goes straight to its pool slot (the
// a2 scatter), the rotated Q row to q_out, so K never makes a second trip
// through HBM.  Pairing: element i with element i + d/2 ("rotate half").
#include <math.h>

#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kMaxThreads = 1024;

// Angles in fixed-point turns.  The host passes, per pair i, the fraction
// F_i / 2^64 = frac(inv_freq_i / (2 pi)) of a turn per position step.  For
// 0 <= p <= 2^31, p * F_i mod 2^64 is the angle's fraction of a turn; its top
// 32 bits are exactly umulhi(p, F_lo) + p * F_hi (mod 2^32), and dropping the
// low word truncates by less than 2^-32 turn.  Read as a signed int32 that
// is the angle reduced to [-pi, pi) in units of 2^-32 turn, exact whatever the
// position -- so no floating-point range reduction and no fp64 arithmetic,
// which runs at a small fraction of the fp32 rate on this part.  A negative
// position is |p| turned the other way.  On [-pi, pi] the hardware sine and
// cosine approximation is within 4e-7 absolute, a few fp32 roundings of the
// rotated value, and keeps the table off the CTA's critical path.
__device__ __forceinline__ float reduced_angle(int pos, uint32_t f_lo, uint32_t f_hi) {
    const uint32_t m = pos < 0 ? 0u - static_cast<uint32_t>(pos) : static_cast<uint32_t>(pos);
    uint32_t turns = __umulhi(m, f_lo) + m * f_hi;
    if (pos < 0) turns = 0u - turns;
    return static_cast<float>(static_cast<int32_t>(turns)) * 1.4629180792671596e-9f;   // 2 pi / 2^32
}

// One CTA per token, one work item per thread: item (row, j) of a Q or K head
// row holds vectors j and j + d/16 (8 pairs, 16 B each side); the items after
// them copy the V row in 16-byte vectors.  Each thread issues its loads first;
// meanwhile threads i < d/2 turn the position into (cos, sin) of pair i, and
// one barrier publishes the table before the rotation.  A negative or
// out-of-pool slot drops the token's K and V items (q is still rotated).
__global__ void __launch_bounds__(kMaxThreads) rope_store_kernel(RopeStoreArgs a, int64_t n_tokens, int* err) {
    __shared__ float2 cs[kMaxRopePairs];
    const int64_t t = blockIdx.x;
    const int half = a.head_dim >> 1;
    const int slot = __ldg(a.slots + t);
    const bool write_kv = slot >= 0 && slot < a.num_slots;
    if (slot >= a.num_slots && threadIdx.x == 0) record_error(err, PKV_DEVERR_SLOT, static_cast<int>(t));
    const int hv = a.head_dim >> 4;
    const int q_items = a.q ? a.num_heads * hv : 0;
    const int rot_items = q_items + (write_kv ? a.num_kv_heads * hv : 0);
    const int v_items = write_kv ? static_cast<int>(a.kv_row >> 3) : 0;
    const int items = rot_items + v_items;
    for (int base = 0; base < items; base += blockDim.x) {
        const int it = base + threadIdx.x;
        const bool rot = it < rot_items;
        const bool is_q = it < q_items;
        int row = 0, j = 0;
        uint4 x1 = make_uint4(0, 0, 0, 0), x2 = x1;
        if (rot) {
            const int rel = is_q ? it : it - q_items;
            row = rel / hv;
            j = rel - row * hv;
            const uint16_t* src = (is_q ? a.q + t * a.q_stride : a.k + t * a.k_stride) +
                                  static_cast<int64_t>(row) * a.head_dim;
            x1 = __ldcs(reinterpret_cast<const uint4*>(src) + j);
            x2 = __ldcs(reinterpret_cast<const uint4*>(src) + j + hv);
        } else if (it < items) {
            j = it - rot_items;
            x1 = __ldcs(reinterpret_cast<const uint4*>(a.v + t * a.v_stride) + j);
        }
        if (base == 0) {
            if (threadIdx.x < half) {
                const uint64_t f = a.turns[threadIdx.x];
                float sn, cn;
                __sincosf(reduced_angle(__ldg(a.positions + t), static_cast<uint32_t>(f),
                                      static_cast<uint32_t>(f >> 32)), &sn, &cn);
                cs[threadIdx.x] = make_float2(cn, sn);
            }
            __syncthreads();
        }
        if (rot) {
            const uint32_t w1[4] = {x1.x, x1.y, x1.z, x1.w};
            const uint32_t w2[4] = {x2.x, x2.y, x2.z, x2.w};
            uint32_t y1[4], y2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 c0 = cs[8 * j + 2 * e], c1 = cs[8 * j + 2 * e + 1];
                const float a0 = bf16_lo(w1[e]), a1 = bf16_hi(w1[e]);
                const float b0 = bf16_lo(w2[e]), b1 = bf16_hi(w2[e]);
                y1[e] = pack_bf16x2(fmaf(a0, c0.x, -b0 * c0.y), fmaf(a1, c1.x, -b1 * c1.y));
                y2[e] = pack_bf16x2(fmaf(b0, c0.x, a0 * c0.y), fmaf(b1, c1.x, a1 * c1.y));
            }
            uint16_t* dst = is_q ? a.q_out + t * a.q_out_stride
                                 : a.k_cache + static_cast<int64_t>(slot) * a.kv_row;
            dst += static_cast<int64_t>(row) * a.head_dim;
            reinterpret_cast<uint4*>(dst)[j] = make_uint4(y1[0], y1[1], y1[2], y1[3]);
            reinterpret_cast<uint4*>(dst)[j + hv] = make_uint4(y2[0], y2[1], y2[2], y2[3]);
        } else if (it < items) {
            reinterpret_cast<uint4*>(a.v_cache + static_cast<int64_t>(slot) * a.kv_row)[j] = x1;
        }
    }
}

// ---------------------------------------------------------------------------
// Staged path (head_dim 128, a token's rows within kMaxStageBytes): persistent
// CTAs, two per SM, walk tokens t = blockIdx.x, + gridDim.x, ...  Per token a
// stage of shared memory holds its Q, K and V rows:
//   warp 0, lane 0   bulk-copies the three rows in (one mbarrier, "full");
//   warps 1-4        rotate Q and K in place, thread (row r, word j) turning
//                    the pairs (2j, 2j+64) and (2j+1, 2j+65) of rows r, r+4,
//                    ... with its own two (cos, sin) -- no table, no CTA
//                    barrier -- then arrive on "rotated";
//   warp 5, lane 0   bulk-stores rotated Q to q_out, rotated K and the
//                    untouched V straight from the stage to the pool slot,
//                    and frees the stage ("empty") once its stores have read it.
// kStages stages per CTA keep ~24 tokens per SM in flight.
// ---------------------------------------------------------------------------
constexpr int kStages = 12;
constexpr int kStoresInFlight = 3;      // store groups still reading their stage
constexpr int kRotWarps = 4;
constexpr int kStagedThreads = 32 * (kRotWarps + 2);
constexpr int kMaxStageBytes = 16384;
// The loader refills a stage only after the store warp releases it, which happens kStoresInFlight
// tokens after that stage's token; with no more stages than that, the loader and the store warp
// would wait on each other.
static_assert(kStages > kStoresInFlight, "the stage ring must be deeper than the stores in flight");

__global__ void __launch_bounds__(kStagedThreads) rope_store_staged_kernel(RopeStoreArgs a, int64_t n_tokens,
                                                                           int* err) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int qb = a.q ? a.num_heads * 256 : 0;          // bytes of the Q rows (d = 128)
    const int kvb = static_cast<int>(a.kv_row) * 2;
    const int stage_bytes = qb + 2 * kvb;
    const uint32_t stage0 = smem_u32(smem);
    const uint32_t bars = stage0 + kStages * stage_bytes;   // full[S], rotated[S], empty[S]
    auto full = [&](int s) { return bars + 8u * s; };
    auto rotated = [&](int s) { return bars + 8u * (kStages + s); };
    auto empty = [&](int s) { return bars + 8u * (2 * kStages + s); };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(rotated(s), 32 * kRotWarps);
            mbar_init(empty(s), 1);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const int64_t first = blockIdx.x;
    const int64_t n_mine = first < n_tokens ? (n_tokens - first + gridDim.x - 1) / gridDim.x : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        if (lane == 0) {
            int64_t i = 0;
            for (; i < n_mine; ++i) {
                const int s = static_cast<int>(i % kStages);
                if (i >= kStages && !mbar_wait(empty(s), static_cast<uint32_t>((i / kStages - 1) & 1), err, 1)) break;
                const int64_t t = first + i * gridDim.x;
                const uint32_t dst = stage0 + s * stage_bytes;
                mbar_arrive_expect_tx(full(s), stage_bytes);
                if (qb) bulk_load(dst, a.q + t * a.q_stride, qb, full(s));
                bulk_load(dst + qb, a.k + t * a.k_stride, kvb, full(s));
                bulk_load(dst + qb + kvb, a.v + t * a.v_stride, kvb, full(s));
            }
            // the last copies must land before the CTA's shared memory goes away (they have by the
            // time the other roles are done; this matters only when a wait above gave up)
            for (int64_t k = i > kStages ? i - kStages : 0; k < i; ++k)
                mbar_wait(full(static_cast<int>(k % kStages)), static_cast<uint32_t>((k / kStages) & 1), err, 2);
        }
    } else if (warp <= kRotWarps) {
        const int ct = threadIdx.x - 32;
        const int j = ct & 31;                  // word j and j + 32 of a 128-element row
        const int r0 = ct >> 5;                 // rows r0, r0 + 4, ...
        const int hq = qb ? a.num_heads : 0;
        const int rows = hq + a.num_kv_heads;
        const uint64_t f0 = a.turns[2 * j], f1 = a.turns[2 * j + 1];
        int pos_win = 0;                        // lane k: position of token i_base + k
        for (int64_t i = 0; i < n_mine; ++i) {
            if ((i & 31) == 0) {                // positions come 32 tokens at a time, off the per-token path
                const int64_t ti = i + lane;
                pos_win = ti < n_mine ? __ldg(a.positions + first + ti * gridDim.x) : 0;
            }
            const int s = static_cast<int>(i % kStages);
            const bool ok = mbar_wait(full(s), static_cast<uint32_t>((i / kStages) & 1), err, 3);
            if (__any_sync(0xffffffffu, !ok)) break;
            const int pos = __shfl_sync(0xffffffffu, pos_win, static_cast<int>(i & 31));
            float s0, c0, s1, c1;
            __sincosf(reduced_angle(pos, static_cast<uint32_t>(f0), static_cast<uint32_t>(f0 >> 32)), &s0, &c0);
            __sincosf(reduced_angle(pos, static_cast<uint32_t>(f1), static_cast<uint32_t>(f1 >> 32)), &s1, &c1);
            uint32_t* st = reinterpret_cast<uint32_t*>(smem + s * stage_bytes);
            for (int r = r0; r < rows; r += kRotWarps) {
                uint32_t* w = st + (r < hq ? r * 64 : (qb >> 2) + (r - hq) * 64);
                const uint32_t x1 = w[j], x2 = w[j + 32];
                const float a0 = bf16_lo(x1), a1 = bf16_hi(x1), b0 = bf16_lo(x2), b1 = bf16_hi(x2);
                w[j] = pack_bf16x2(fmaf(a0, c0, -b0 * s0), fmaf(a1, c1, -b1 * s1));
                w[j + 32] = pack_bf16x2(fmaf(b0, c0, a0 * s0), fmaf(b1, c1, a1 * s1));
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the bulk stores
            mbar_arrive(rotated(s));
        }
    } else {
        // the whole warp walks the tokens (slots come 32 at a time, one per lane); lane 0 stores
        int slot_win = -1;
        for (int64_t i = 0; i < n_mine; ++i) {
            if ((i & 31) == 0) {
                const int64_t ti = i + lane;
                slot_win = ti < n_mine ? __ldg(a.slots + first + ti * gridDim.x) : -1;
            }
            const int s = static_cast<int>(i % kStages);
            const bool ok = mbar_wait(rotated(s), static_cast<uint32_t>((i / kStages) & 1), err, 4);
            if (__any_sync(0xffffffffu, !ok)) break;
            const int slot = __shfl_sync(0xffffffffu, slot_win, static_cast<int>(i & 31));
            if (lane != 0) continue;
            const int64_t t = first + i * gridDim.x;
            const uint32_t src = stage0 + s * stage_bytes;
            if (qb) bulk_store(a.q_out + t * a.q_out_stride, src, qb);
            if (slot >= 0 && slot < a.num_slots) {
                bulk_store(a.k_cache + static_cast<int64_t>(slot) * a.kv_row, src + qb, kvb);
                bulk_store(a.v_cache + static_cast<int64_t>(slot) * a.kv_row, src + qb + kvb, kvb);
            } else if (slot >= a.num_slots) {
                record_error(err, PKV_DEVERR_SLOT, static_cast<int>(t));
            }
            bulk_commit();
            bulk_wait_read<kStoresInFlight>();    // token i - kStoresInFlight's stores have read their stage
            if (i >= kStoresInFlight) mbar_arrive(empty(static_cast<int>((i - kStoresInFlight) % kStages)));
        }
        if (lane == 0) bulk_wait<0>();           // all stores done before the shared memory is released
    }
}

}  // namespace

int rope_store_threads(const RopeStoreArgs& a) {
    const int64_t hv = a.head_dim / 16;
    const int64_t items = (a.q ? a.num_heads : 0) * hv + a.num_kv_heads * hv + a.kv_row / 8;
    const int64_t threads = std::max<int64_t>((items + 31) / 32 * 32, a.head_dim / 2);
    return threads > kMaxThreads ? 0 : static_cast<int>(threads);
}

cudaError_t launch_rope_store(const RopeStoreArgs& a, int64_t n_tokens, int* err, cudaStream_t stream) {
    if (n_tokens == 0) return cudaSuccess;
    const int64_t stage = (a.q ? a.num_heads * 256 : 0) + 4 * a.kv_row;
    if (a.head_dim == 128 && stage <= kMaxStageBytes) {
        const size_t smem = static_cast<size_t>(kStages) * stage + 3 * kStages * 8;
        if (!setup_once(kSetupRopeStore, [] {
                return cudaFuncSetAttribute(rope_store_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(kStages * kMaxStageBytes + 3 * kStages * 8)) ==
                       cudaSuccess;
            }))
            return cudaErrorUnknown;
        const int64_t grid = std::min<int64_t>(n_tokens, 2LL * sm_count());
        rope_store_staged_kernel<<<static_cast<unsigned>(grid), kStagedThreads, smem, stream>>>(a, n_tokens, err);
        return cudaGetLastError();
    }
    const int threads = rope_store_threads(a);
    const int64_t grid = n_tokens;
    rope_store_kernel<<<static_cast<unsigned>(grid), threads, 0, stream>>>(a, n_tokens, err);
    return cudaGetLastError();
}

}  // namespace pkv
