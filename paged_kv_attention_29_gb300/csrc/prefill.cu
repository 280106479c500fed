// a3: varlen prefill attention over the paged KV cache, on tcgen05 tensor cores.
//
// Visual atlas (diomchen.github.io/reference/visual-atlas.html): figure
// "cu_seqlens=[0,3,5]" (packed requests), figs. 16-17 (softmax(scale QK^T +
// mask) V, diagonal kept, a cached chunk keeps its position offset: query i
// of a chunk sees keys j <= i + k_len - q_len), fig. 18 (two query heads share
// a K/V head), fig. 22 (blockwise evaluation without materialising scores).
//
// One CTA computes a 128-row tile: 64 query tokens x the 2 query heads that
// share KV head g.  Packing both heads into the MMA's M dimension means both
// read the same K/V tile, loaded once, with no cross-CTA traffic.
//
//   Q tile   smem, two 128B-swizzled boxes (head dims 0-63, 64-127), rows in
//            (token, head) order straight from the [tokens, heads, 128] layout
//   K, V     128 keys (half of a 256-token block) per tile, two boxes each,
//            double-buffered; cut from the pool by a 4-D tensor map at the
//            physical block the block table names
//   S = QK^T tcgen05.mma M=128 N=128 K=16 x 8, fp32 in TMEM (two buffers)
//   P        bf16, written back to TMEM over its own S buffer; O += P V with P
//            as the TMEM A operand and V as an MN-major smem B operand
//   O        fp32 in TMEM; rescaled only when a row max grows by more than
//            2^8 (the stale max keeps exp2 below 256, and O and l share it)
//
// Warp roles: warps 0-3 own TMEM lanes 0-127 (one row each: mask, online
// softmax, O rescale, epilogue); warp 4 issues TMA; warp 5 allocates TMEM and
// one of its lanes issues every MMA.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int D = kHeadDim;
constexpr int G = kGroup;
constexpr int QTOK = 64;                  // query tokens per tile (x G heads = 128 rows)
constexpr int ROWS = QTOK * G;            // MMA M
constexpr int KT = 128;                   // keys per KV tile (MMA N of QK^T)
constexpr int HALF_BYTES = ROWS * 64 * 2; // one 128B-swizzled box: 128 rows x 64 dims = 16 KiB
constexpr int TILE_BYTES = 2 * HALF_BYTES;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int S_COL0 = 0, S_COL1 = 128, O_COL = 256;
constexpr float kRescaleLog2 = 8.0f;

// shared-memory layout (offsets from the 1024-aligned base)
constexpr int SM_Q = 0;
constexpr int SM_K = SM_Q + TILE_BYTES;           // 2 stages
constexpr int SM_V = SM_K + 2 * TILE_BYTES;       // 2 stages
constexpr int SM_BAR = SM_V + 2 * TILE_BYTES;
// barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done,
// o_final (the last PV landed), drain (every MMA landed)
constexpr int BAR_Q = 0, BAR_KF = 1, BAR_KE = 3, BAR_VF = 5, BAR_VE = 7, BAR_SF = 9, BAR_PF = 11,
              BAR_PV = 13, BAR_OFIN = 14, BAR_DRAIN = 15, NUM_BARS = 16;
constexpr int SM_MISC = SM_BAR + NUM_BARS * 8;   // tmem base (u32), abort flag (u32)
constexpr int SMEM_BYTES = SM_MISC + 16 + 1024;  // + alignment slack

struct Params {
    const int32_t* cu_q;
    const int32_t* cu_k;
    const int32_t* block_tables;
    uint16_t* out;
    int max_blocks;
    int num_heads;
    int block_size;
    int num_blocks;
    int n_qtiles;
    float scale_log2;
    int* err;
};

struct Ctl {
    volatile uint32_t* abort;
    int* err;
    int where;
};

// Wait for a phase; any role's timeout aborts the whole CTA.
__device__ __noinline__ bool wait_phase(const Ctl& c, uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *c.abort = 1u;
            record_error(c.err, PKV_DEVERR_TIMEOUT, c.where);
            return false;
        }
    }
}

// Wait used while draining after an abort: bounded, ignores the abort flag.
__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t addr) {
    // 128B swizzle, K-major: rows of 128 B, 8-row atoms 1024 B apart (LBO unused)
    return smem_desc(addr, 16, 1024, 2);
}
__device__ __forceinline__ uint64_t vmajor_desc(uint32_t addr) {
    // 128B swizzle, MN-major (V as [keys][dims]): the second 64-dim box is
    // HALF_BYTES further (LBO), 8-key groups are 1024 B apart (SBO)
    return smem_desc(addr, HALF_BYTES, 1024, 2);
}

__global__ void __launch_bounds__(THREADS, 1)
prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const int seq = blockIdx.z;
    const int g = blockIdx.y;
    const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x);   // heavier tiles first
    const int q_start = __ldg(p.cu_q + seq);
    const int ql = __ldg(p.cu_q + seq + 1) - q_start;
    const int kl = __ldg(p.cu_k + seq + 1) - __ldg(p.cu_k + seq);
    if (qt * QTOK >= ql) return;
    if (ql > kl || kl > p.max_blocks * p.block_size) {
        if (threadIdx.x == 0) record_error(p.err, PKV_DEVERR_SEQLENS, seq);
        return;
    }
    const int offset = kl - ql;
    const int last_q = min(qt * QTOK + QTOK, ql) - 1;
    const int keys_needed = last_q + offset + 1;              // <= kl
    const int n_kv = (keys_needed + KT - 1) / KT;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + SM_Q, sK = base + SM_K, sV = base + SM_V;
    const uint32_t bars = base + SM_BAR;
    auto bar = [&](int i) { return bars + 8u * i; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + SM_MISC);
    Ctl ctl{reinterpret_cast<volatile uint32_t*>(misc + 1), p.err, seq};

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (tid == 0) {
        mbar_init(bar(BAR_Q), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(BAR_KF + s), 1);
            mbar_init(bar(BAR_KE + s), 1);
            mbar_init(bar(BAR_VF + s), 1);
            mbar_init(bar(BAR_VE + s), 1);
            mbar_init(bar(BAR_SF + s), 1);
            mbar_init(bar(BAR_PF + s), ROWS);
        }
        mbar_init(bar(BAR_PV), 1);
        mbar_init(bar(BAR_OFIN), 1);
        mbar_init(bar(BAR_DRAIN), 1);
        misc[1] = 0u;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(base + SM_MISC, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 4) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const int qrow = q_start + qt * QTOK;
            mbar_arrive_expect_tx(bar(BAR_Q), TILE_BYTES);
            tma_load_3d(sQ, &tm_q, bar(BAR_Q), 0, G * g, qrow);
            tma_load_3d(sQ + HALF_BYTES, &tm_q, bar(BAR_Q), 64, G * g, qrow);
            const int32_t* bt = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks;
            int issued_k = 0, issued_v = 0;
            bool ok = true;
            for (int j = 0; j < n_kv && ok; ++j) {
                const int st = j & 1;
                const int key0 = j * KT;
                const int lb = key0 / p.block_size;
                const int phys = __ldg(bt + lb);
                if (phys < 0 || phys >= p.num_blocks) record_error(p.err, PKV_DEVERR_BLOCK_ID, seq);
                const int off = key0 - lb * p.block_size;
                if (j >= 2 && !(ok = wait_phase(ctl, bar(BAR_KE + st), ((j - 2) >> 1) & 1))) break;
                mbar_arrive_expect_tx(bar(BAR_KF + st), TILE_BYTES);
                tma_load_4d(sK + st * TILE_BYTES, &tm_k, bar(BAR_KF + st), 0, g, off, phys);
                tma_load_4d(sK + st * TILE_BYTES + HALF_BYTES, &tm_k, bar(BAR_KF + st), 64, g, off, phys);
                ++issued_k;
                if (j >= 2 && !(ok = wait_phase(ctl, bar(BAR_VE + st), ((j - 2) >> 1) & 1))) break;
                mbar_arrive_expect_tx(bar(BAR_VF + st), TILE_BYTES);
                tma_load_4d(sV + st * TILE_BYTES, &tm_v, bar(BAR_VF + st), 0, g, off, phys);
                tma_load_4d(sV + st * TILE_BYTES + HALF_BYTES, &tm_v, bar(BAR_VF + st), 64, g, off, phys);
                ++issued_v;
            }
            if (*ctl.abort) {
                // let every copy already issued land before shared memory is released
                wait_drain(bar(BAR_Q), 0);
                for (int j = max(0, issued_k - 2); j < issued_k; ++j) wait_drain(bar(BAR_KF + (j & 1)), (j >> 1) & 1);
                for (int j = max(0, issued_v - 2); j < issued_v; ++j) wait_drain(bar(BAR_VF + (j & 1)), (j >> 1) & 1);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(ROWS, KT, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(ROWS, D, 0, 1);
            bool ok = wait_phase(ctl, bar(BAR_Q), 0);
            auto issue_pv = [&](int jj) -> bool {
                const int st = jj & 1;
                if (!wait_phase(ctl, bar(BAR_PF + st), (jj >> 1) & 1)) return false;
                if (!wait_phase(ctl, bar(BAR_VF + st), (jj >> 1) & 1)) return false;
                tc_fence_after();
                const int keys_here = min(KT, kl - jj * KT);
                const int ksteps = (keys_here + 15) >> 4;
                const int tail = keys_here & 15;
                if (tail) {
                    // rows past the sequence's last key may hold anything (freed blocks are
                    // not cleared); P is zero there but 0 * NaN is NaN, so clear them
                    uint8_t* vt = gbase + SM_V + st * TILE_BYTES;
                    for (int r = keys_here; r < ksteps * 16; ++r) {
                        uint4* r0 = reinterpret_cast<uint4*>(vt + r * 128);
                        uint4* r1 = reinterpret_cast<uint4*>(vt + HALF_BYTES + r * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) { r0[c] = make_uint4(0, 0, 0, 0); r1[c] = make_uint4(0, 0, 0, 0); }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                const uint32_t p_tmem = tmem + (st ? S_COL1 : S_COL0);
                const uint32_t vbase = sV + st * TILE_BYTES;
                for (int ks = 0; ks < ksteps; ++ks) {
                    mma_ts(tmem + O_COL, p_tmem + ks * 8, vmajor_desc(vbase + ks * 16 * 128), idesc_pv,
                           (jj > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(bar(BAR_PV));
                mma_commit(bar(BAR_VE + st));
                return true;
            };
            for (int j = 0; j < n_kv && ok; ++j) {
                const int st = j & 1;
                if (!(ok = wait_phase(ctl, bar(BAR_KF + st), (j >> 1) & 1))) break;
                tc_fence_after();
                const uint32_t kbase = sK + st * TILE_BYTES;
                const uint32_t s_tmem = tmem + (st ? S_COL1 : S_COL0);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t koff = (ks >> 2) * HALF_BYTES + (ks & 3) * 32;
                    mma_ss(s_tmem, kmajor_desc(sQ + koff), kmajor_desc(kbase + koff), idesc_qk, ks > 0 ? 1u : 0u);
                }
                mma_commit(bar(BAR_SF + st));
                mma_commit(bar(BAR_KE + st));
                if (j >= 1 && !(ok = issue_pv(j - 1))) break;
            }
            if (ok) ok = issue_pv(n_kv - 1);
            if (ok) mma_commit(bar(BAR_OFIN));
            // everything issued has to finish before TMEM is released
            mma_commit(bar(BAR_DRAIN));
            wait_drain(bar(BAR_DRAIN), 0);
        }
    } else {
        // ------------------------------------------------------------ softmax rows
        const int row = tid;                       // TMEM lane
        const int ti = row >> 1;
        const int hh = row & 1;
        const int qi = qt * QTOK + ti;
        const bool row_valid = qi < ql;
        const int jmax = min(qi + offset, kl - 1);   // last visible key
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int st = j & 1;
            ok = __all_sync(0xffffffffu, wait_phase(ctl, bar(BAR_SF + st), (j >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            const uint32_t s_tmem = tmem + lane_off + (st ? S_COL1 : S_COL0);
            uint32_t s[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + 32 * c, s[c]);
            tmem_ld_wait();
            const int lim = jmax - j * KT;         // columns <= lim are visible
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float x = (32 * c + e <= lim) ? __uint_as_float(s[c][e]) * p.scale_log2 : -INFINITY;
                    s[c][e] = __float_as_uint(x);
                    mt = fmaxf(mt, x);
                }
            const float m_new = fmaxf(m_used, mt);
            if (j == 0) {
                m_used = m_new;
            } else {
                const bool need = m_new > m_used + kRescaleLog2;
                if (__any_sync(0xffffffffu, need)) {
                    // O holds sum_{k<j} P_k V_k scaled by 2^-m_used; PV_{j-1} must have landed.
                    // S_j landing implies PV_{j-2} landed (one commit tracks all earlier MMAs),
                    // so the phase parity of PV_{j-1} cannot alias.
                    ok = __all_sync(0xffffffffu, wait_phase(ctl, bar(BAR_PV), (j - 1) & 1));
                    if (!ok) break;
                    tc_fence_after();
                    const float m_tgt = fmaxf(m_used, m_new);
                    const float alpha = exp2f(m_used - m_tgt);
                    const uint32_t o_tmem = tmem + lane_off + O_COL;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(o_tmem + 32 * c, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(o_tmem + 32 * c, o);
                    }
                    tmem_st_wait();
                    l *= alpha;
                    m_used = m_tgt;
                }
            }
            // P = 2^(x - m_used) in bf16, over this tile's S buffer
            uint32_t pk[2][32];
            float rs = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float p0 = exp2f(__uint_as_float(s[c][e]) - m_used);
                    const float p1 = exp2f(__uint_as_float(s[c][e + 1]) - m_used);
                    rs += p0 + p1;
                    pk[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_bf16x2(p0, p1);
                }
            l += rs;
            tmem_st32(s_tmem, pk[0]);
            tmem_st32(s_tmem + 32, pk[1]);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(BAR_PF + st));
        }
        // epilogue: O / l -> bf16
        if (ok) ok = __all_sync(0xffffffffu, wait_phase(ctl, bar(BAR_OFIN), 0));
        if (ok) {
            tc_fence_after();
            const uint32_t o_tmem = tmem + lane_off + O_COL;
            const float inv = 1.f / l;
            uint16_t* dst = p.out + (static_cast<int64_t>(q_start + qi) * p.num_heads + G * g + hh) * D;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(o_tmem + 32 * c, o);
                tmem_ld_wait();
                if (row_valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
                        d4[v] = w;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

pkv_status launch_prefill(const PrefillArgs& a, int* err, cudaStream_t stream) {
    if (a.num_seqs == 0 || a.total_q == 0 || a.max_seqlen_q == 0) return PKV_OK;
    CUtensorMap tm_q, tm_k, tm_v;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_heads),
                                  static_cast<uint64_t>(a.total_q)};
        const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.num_heads) * D * 2};
        const uint32_t box[3] = {64u, static_cast<uint32_t>(G), static_cast<uint32_t>(QTOK)};
        if (encode_tiled(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.q), dims, strides,
                         box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return PKV_ERR_INVALID_ARG;
    }
    {
        const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_kv_heads),
                                  static_cast<uint64_t>(a.block_size), static_cast<uint64_t>(a.num_blocks)};
        const uint64_t strides[3] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.num_kv_heads) * D * 2,
                                     static_cast<uint64_t>(a.block_size) * a.num_kv_heads * D * 2};
        const uint32_t box[4] = {64u, 1u, static_cast<uint32_t>(KT), 1u};
        if (encode_tiled(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(a.k_cache), dims,
                         strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return PKV_ERR_INVALID_ARG;
        if (encode_tiled(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(a.v_cache), dims,
                         strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return PKV_ERR_INVALID_ARG;
    }
    Params p;
    p.cu_q = a.cu_q;
    p.cu_k = a.cu_k;
    p.block_tables = a.block_tables;
    p.out = a.out;
    p.max_blocks = a.max_blocks;
    p.num_heads = a.num_heads;
    p.block_size = a.block_size;
    p.num_blocks = a.num_blocks;
    p.n_qtiles = (a.max_seqlen_q + QTOK - 1) / QTOK;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    p.err = err;

    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(prefill_tcgen05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured_device = dev;
    }
    dim3 grid(p.n_qtiles, a.num_kv_heads, a.num_seqs);
    prefill_tcgen05_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(tm_q, tm_k, tm_v, p);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
