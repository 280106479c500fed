// a3: varlen prefill attention over the paged KV cache, on tcgen05 tensor cores.
//
// Visual atlas (diomchen.github.io/reference/visual-atlas.html): figure
// "cu_seqlens=[0,3,5]" (packed requests), figs. 16-17 (softmax(scale QK^T +
// mask) V, diagonal kept, a cached chunk keeps its position offset: query i
// of a chunk sees keys j <= i + k_len - q_len), fig. 18 (two query heads share
// a K/V head), fig. 22 (blockwise evaluation without materialising scores).
//
// Work unit: 256 / G query tokens of one sequence x one KV head g, split into
// two 128-row tiles A and B (128 / G tokens x the G query heads of the group
// each, so all G heads read one K/V tile; G = num_heads / num_kv_heads is 1, 2,
// 4 or 8, row r of a tile being token r / G, head G g + r % G).  Per unit and
// 128-key tile j:
//
//   S_X(j) = Q_X K_j^T      tcgen05.mma M=128 N=128, 8 x K=16, fp32 in TMEM
//   P_X(j)                  masked online softmax by warpgroup X, bf16 over S_X
//   O_X   += P_X(j) V_j     tcgen05.mma with P from TMEM (A operand), V MN-major
//
// The MMA warp issues S_A(0) S_B(0) | PV_A(0) S_A(1) PV_B(0) S_B(1) | ... so
// the tensor core works on one tile while the other tile's warpgroup runs its
// softmax.  Because one commit tracks every earlier MMA, S_X(j) landing means
// PV_X(j-1) landed, so a warpgroup may rescale O_X after it sees S_X(j) with
// no further wait; O is rescaled only when a row max grows by more than 2^8
// (P then stays below 256, and O and the row sum share the stale max).
//
// The softmax warps' code is kept small: two softmax warps share each
// scheduler, and rolling the rare rescale loop and the epilogue's outer loop
// (no spills left) took a call from 54.9 to 51.9 us, bit-identical.
//
// The softmax is the critical path, so it is written for the fewest issued
// instructions per score: one 3-input max per two scores, the exponent
// argument as one packed fp32x2 FMA per two scores, one special-function
// exp2, a packed fp32x2 add for the row sum and one bf16x2 pack per two; the
// mask is applied only on tiles the diagonal crosses.
//
// Persistent CTAs (one per SM) take units from a list that a one-CTA plan
// kernel sorts by cost (the longer tile's KV tiles, costliest first) and leaves
// in the workspace: CTA i starts with unit i, and each CTA's producer claims
// its next unit with an atomic increment when its current unit starts.  The
// plan's scan over cost buckets runs on a warp, 32 buckets per step.  The two
// launches are chained with
// programmatic dependent launch so this kernel's set-up overlaps the plan.
//
// Warps 0-3: softmax of tile A (TMEM lanes 0-127), warps 4-7: tile B; warp 8:
// TMA producer; warp 9: TMEM allocation and MMA issue (the whole warp runs the
// loop, one lane elected per tcgen05 instruction); warps 10-11 only complete
// the third warpgroup for the register split.
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int D = kHeadDim;
constexpr int ROWS = 128;                 // MMA M: rows of a tile, (128 / G tokens) x (G heads)
constexpr int KT = 128;                   // keys per KV tile
constexpr int HALF_BYTES = ROWS * 64 * 2; // one 128B-swizzled box: 128 rows x 64 dims = 16 KiB
constexpr int TILE_BYTES = 2 * HALF_BYTES;
constexpr int THREADS = 384;              // 3 warpgroups: softmax A, softmax B, producer + MMA
constexpr int PRODUCER_WARP = 8, MMA_WARP = 9;
// setmaxnreg split: the softmax warpgroups keep a 128-column fp32 S row per
// thread; the control warpgroup needs few.  2*128*208 + 128*80 = 63488
// registers, within the 384 x 168 that the launch must provide (checked on
// the host before every launch).
constexpr uint32_t kSoftmaxRegs = 208, kControlRegs = 80, kMinLaunchRegs = 168;
constexpr int TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t S_COL(int x) { return 128u * x; }         // S / P of tile x
__host__ __device__ constexpr uint32_t O_COL(int x) { return 256u + 128u * x; }  // O of tile x
constexpr float kRescaleLog2 = 8.0f;

// shared memory (offsets from the 1024-aligned base)
constexpr int SM_QA = 0;
constexpr int SM_QB = SM_QA + TILE_BYTES;
constexpr int SM_K = SM_QB + TILE_BYTES;          // 2 stages
constexpr int SM_V = SM_K + 2 * TILE_BYTES;       // 2 stages
constexpr int SM_STAGE = SM_V + 2 * TILE_BYTES;   // epilogue staging: 4 KiB per softmax warp
constexpr int STAGE_WARP_BYTES = 32 * 128;
constexpr int SM_BAR = SM_STAGE + 8 * STAGE_WARP_BYTES;
constexpr int RING = 4;                           // unit ring: producer -> MMA and softmax warps
enum {
    BAR_QF = 0, BAR_QE, BAR_GF, BAR_GF1, BAR_GE, BAR_GE1, BAR_SF, BAR_SF1, BAR_PF, BAR_PF1, BAR_OF, BAR_OF1, BAR_OE, BAR_OE1, BAR_DRAIN,
    BAR_UF, BAR_UE = BAR_UF + RING, NUM_BARS = BAR_UE + RING
};
constexpr int RING_READERS = 1 + 8;               // the MMA thread and one lane of each softmax warp
constexpr int SM_RING = (SM_BAR + NUM_BARS * 8 + 31) & ~31;   // RING x {idx, record}: 16-byte fields
constexpr int SM_MISC = SM_RING + RING * 32;      // [0] TMEM base, [1] abort flag
constexpr int SMEM_BYTES = SM_MISC + 16 + 1024;
static_assert(SM_QA % 1024 == 0 && SM_QB % 1024 == 0 && SM_K % 1024 == 0 && SM_V % 1024 == 0,
              "128B-swizzled operand tiles need 1024-byte alignment");
static_assert(SM_STAGE % 16 == 0 && SM_BAR % 8 == 0 && SM_RING % 16 == 0 && SM_MISC % 16 == 0,
              "vector, barrier and ring fields need their natural alignment");

struct Params {
    const int32_t* cu_q;
    const int32_t* cu_k;
    const int32_t* block_tables;
    const uint4* plan;        // [0] = {number of (seq, pair) records, unit counter, 0, tag};
                              // then {seq << 16 | pair, q_start, q_len, k_len}, costliest first
    unsigned int* next_unit;  // &plan[0].y: units from gridDim.x on are taken in list order by atomic increments
    uint16_t* out;
    int max_blocks;
    int num_heads;
    int num_kv_heads;
    int lg;                   // log2 of the group size G
    int block_size;
    int num_blocks;
    float scale_log2;
    uint32_t tag;             // the plan this launch expects (see plan_tag)
    int* err;
};

struct Ctl {
    volatile uint32_t* abort;
    int* err;
};

// Inlined on purpose: a call inside a setmaxnreg region cannot be register-allocated.
// A waiting thread sleeps in try_wait (up to ~0.5 ms per try) instead of
// spinning, so the warps it shares a scheduler with -- the MMA-issuing and
// TMA warps -- keep their issue slots.
__device__ __forceinline__ bool wait_phase(const Ctl& c, uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 500000u)) return true;
        if (*c.abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *c.abort = 1u;
            record_error(c.err, PKV_DEVERR_TIMEOUT, static_cast<int>(blockIdx.x));
            return false;
        }
    }
}

// wait_phase for a warp that runs in step: every lane waits, and the result is
// made warp-uniform.
__device__ __forceinline__ bool wait_warp(const Ctl& c, uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_phase(c, bar, parity));
}

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_sleep(bar, parity, 500000u))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t addr) { return smem_desc(addr, 16, 1024, 2); }
__device__ __forceinline__ uint64_t vmajor_desc(uint32_t addr) { return smem_desc(addr, HALF_BYTES, 1024, 2); }

// KV tiles a query tile of qtok tokens needs: keys up to its last token's position.
__device__ __forceinline__ int kv_tiles(int first_tok, int qtok, int ql, int offset) {
    if (first_tok >= ql) return 0;
    const int last = min(first_tok + qtok, ql) - 1;
    return (last + offset + KT) / KT;     // ceil((last + offset + 1) / KT)
}

struct Unit {
    int seq, pair, g;
    int q_start, ql, kl, offset;
    int n[2];          // KV tiles of tile A and tile B (B may be 0)
};

// One 16-byte record per (seq, pair), so a unit's metadata is a single load that
// can be issued a whole unit ahead of its use.
__device__ __forceinline__ uint4 unit_record(const Params& p, int idx) {
    return idx >= 0 ? __ldg(p.plan + 1 + idx / p.num_kv_heads) : make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ Unit unit_from(const Params& p, int idx, uint4 rec) {
    Unit u;
    u.g = idx % p.num_kv_heads;
    u.seq = static_cast<int>(rec.x >> 16);
    u.pair = static_cast<int>(rec.x & 0xffffu);
    u.q_start = static_cast<int>(rec.y);
    u.ql = static_cast<int>(rec.z);
    u.kl = static_cast<int>(rec.w);
    u.offset = u.kl - u.ql;
    const int qtok = ROWS >> p.lg;
    u.n[0] = kv_tiles(u.pair * 2 * qtok, qtok, u.ql, u.offset);
    u.n[1] = kv_tiles(u.pair * 2 * qtok + qtok, qtok, u.ql, u.offset);
    return u;
}

// Next unit of the cost-sorted list for this CTA, or -1: CTA i starts with unit i,
// and after that CTAs take units in list order as they free up (longest first,
// so the last units to start are the shortest and the CTAs finish close together).
// Every CTA that starts with a unit grabs until one grab fails, so one call makes exactly
// `total` grabs; the last of them resets the counter, which leaves the plan ready for the
// next call on it.  The reset sits in a CTA's last look-ahead, not at the kernel's end.
__device__ __forceinline__ int grab_unit(const Params& p, int total) {
    const unsigned int v = atomicAdd(p.next_unit, 1u);
    if (v == static_cast<unsigned int>(total) - 1u) atomicExch(p.next_unit, 0u);
    const int idx = static_cast<int>(v + gridDim.x);
    return idx < total ? idx : -1;
}

// The producer hands every unit (index and record) to the MMA thread and the
// softmax warps through a ring in shared memory: slot r % RING, "full" barrier
// (one arrival) and "empty" barrier (RING_READERS arrivals).
struct alignas(16) RingEntry {
    int idx;
    int pad[3];
    uint4 rec;
};
static_assert(sizeof(RingEntry) == 32, "ring slots are 32 bytes");

// -------------------------------------------------------------------------
// plan: (seq, pair) entries sorted by cost, most expensive first
//
// Tiles A and B of a unit run in lockstep (the MMA warp alternates between them and
// each has its own softmax warpgroup), so a unit takes about as long as its longer
// tile, plus a little when B exists: measured per unit, a lone 8-tile A takes
// 13.7 us against 8.7 us for 4 + 4 tiles.  The cost is therefore 2 max(nA, nB),
// plus 1 when B exists (B never has fewer tiles than A).
__device__ __forceinline__ int unit_cost(int pr, int qtok, int ql, int off) {
    const int na = kv_tiles(pr * 2 * qtok, qtok, ql, off), nb = kv_tiles(pr * 2 * qtok + qtok, qtok, ql, off);
    return 2 * max(na, nb) + (nb > 0 ? 1 : 0);
}
// -------------------------------------------------------------------------
__global__ void __launch_bounds__(256) prefill_plan_kernel(const int32_t* __restrict__ cu_q,
                                                           const int32_t* __restrict__ cu_k, int num_seqs,
                                                           int total_q, int max_blocks, int block_size, int qtok,
                                                           int max_cost, uint32_t tag, uint4* __restrict__ plan,
                                                           int* err) {
    extern __shared__ int hist[];          // [max_cost + 1]
    const int unit_tok = 2 * qtok;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = threadIdx.x; i <= max_cost; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    auto seq_ok = [&](int s, int& ql, int& kl) {
        const int q0 = cu_q[s], q1 = cu_q[s + 1];
        ql = q1 - q0;
        kl = cu_k[s + 1] - cu_k[s];
        return q0 >= 0 && q1 <= total_q && ql >= 0 && ql <= kl && kl <= max_blocks * block_size;
    };
    for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
        int ql, kl;
        if (!seq_ok(s, ql, kl)) {
            record_error(err, PKV_DEVERR_SEQLENS, s);
            continue;
        }
        const int off = kl - ql;
        for (int pr = 0; pr * unit_tok < ql; ++pr) {
            const int cost = min(max_cost, unit_cost(pr, qtok, ql, off));
            atomicAdd(&hist[cost], 1);
        }
    }
    __syncthreads();
    // exclusive scan in descending cost order (costliest first), 32 buckets per step of warp 0
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int run = 0;
        for (int top = max_cost; top >= 0; top -= 32) {
            const int c = top - lane;
            const int x = c >= 0 ? hist[c] : 0;
            int incl = x;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            if (c >= 0) hist[c] = run + incl - x;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) plan[0] = make_uint4(static_cast<uint32_t>(run), 0u, 0u, tag);
    }
    __syncthreads();
    for (int s = threadIdx.x; s < num_seqs; s += blockDim.x) {
        int ql, kl;
        if (!seq_ok(s, ql, kl)) continue;
        const int off = kl - ql;
        for (int pr = 0; pr * unit_tok < ql; ++pr) {
            const int cost = min(max_cost, unit_cost(pr, qtok, ql, off));
            const int pos = atomicAdd(&hist[cost], 1);
            plan[1 + pos] = make_uint4((static_cast<uint32_t>(s) << 16) | static_cast<uint32_t>(pr),
                                       static_cast<uint32_t>(cu_q[s]), static_cast<uint32_t>(ql),
                                       static_cast<uint32_t>(kl));
        }
    }
}

// -------------------------------------------------------------------------
// main kernel
// -------------------------------------------------------------------------
__global__ void __launch_bounds__(THREADS, 1)
prefill_fa_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sQ[2] = {base + SM_QA, base + SM_QB};
    const uint32_t sK = base + SM_K, sV = base + SM_V;
    const uint32_t bars = base + SM_BAR;
    auto bar = [&](int i) { return bars + 8u * i; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + SM_MISC);
    RingEntry* ring = reinterpret_cast<RingEntry*>(gbase + SM_RING);
    Ctl ctl{reinterpret_cast<volatile uint32_t*>(misc + 1), p.err};

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < NUM_BARS; ++i) {
            const bool softmax_arrive = (i == BAR_PF || i == BAR_PF1 || i == BAR_OE || i == BAR_OE1);
            const bool ring_empty = i >= BAR_UE && i < BAR_UE + RING;
            mbar_init(bar(i), softmax_arrive ? ROWS : ring_empty ? RING_READERS : 1);
        }
        misc[1] = 0u;
        fence_barrier_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(base + SM_MISC, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // everything above overlaps the plan kernel; global reads start here
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Each warpgroup runs its own branch to the kernel's end (no common tail, so
    // every instruction has one register budget); every branch ends at the same
    // CTA barrier, after which the MMA warp releases TMEM.
    if (warp == PRODUCER_WARP) {
        regs_dec<kControlRegs>();
        // ---------------------------------------------------------------- TMA
        if (lane == 0) {
            // The plan's header and this CTA's first record, read together (one round trip; the
            // record of unit blockIdx.x lies inside the workspace whatever the header says).  A
            // plan made for other lengths, bounds or group size is not used: nothing is computed.
            const uint4 head = __ldcg(p.plan);
            const uint4 rec_first = __ldcg(p.plan + 1 + blockIdx.x / p.num_kv_heads);
            const bool plan_ok = head.w == p.tag;
            if (!plan_ok && blockIdx.x == 0) record_error(p.err, PKV_DEVERR_PLAN, 0);
            const int total_units = plan_ok ? static_cast<int>(head.x) * p.num_kv_heads : 0;
            int uq = 0, groups = 0;   // Q tiles and K/V groups issued
            // a tile's K or V: TMA from the physical block the table names (128 keys, two 64-dim halves)
            // where tile jj of unit w lives: its physical block (from the block table) and the offset
            // of its first key in that block
            struct Loc {
                int phys, off, g;
            };
            auto locate = [&](const Unit& w, int jj) {
                const int key0 = jj * KT;
                const int lb = key0 / p.block_size;
                Loc l;
                l.phys = __ldg(p.block_tables + static_cast<int64_t>(w.seq) * p.max_blocks + lb);
                if (l.phys < 0 || l.phys >= p.num_blocks) record_error(p.err, PKV_DEVERR_BLOCK_ID, w.seq);
                l.off = key0 - lb * p.block_size;
                l.g = w.g;
                return l;
            };
            auto load_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t b, const Loc& l) {
                tma_load_4d(dst, map, b, 0, l.g, l.off, l.phys);
                tma_load_4d(dst + HALF_BYTES, map, b, 64, l.g, l.off, l.phys);
            };
            // A group's V tile is the tile whose K went into the group before, so its block is known;
            // the K tile's block is looked up one group early, after the previous group's copies are
            // issued, so no block-table load sits between a stage's release and its refill.
            Loc k_at = {0, 0, 0};                     // the tile of the last K copy
            Loc pref = {0, 0, 0};
            int pref_idx = -2, pref_tile = -1;        // what `pref` locates
            // one unit of lookahead: the next unit is taken when the current one starts (its first K
            // tile rides in the current unit's last group), so no CTA holds more than one unit it
            // has not started.  The first unit of CTA i is unit i (no atomic round trip before the
            // first copies); the queue hands out the rest from unit gridDim.x on.
            int idx_cur = static_cast<int>(blockIdx.x) < total_units ? static_cast<int>(blockIdx.x) : -1;
            uint4 rec_cur = idx_cur >= 0 ? rec_first : make_uint4(0u, 0u, 0u, 0u);
            bool owe_grab = idx_cur >= 0;             // this CTA has yet to make its failing grab
            bool ok = true;
            if (idx_cur >= 0) {                       // group 0: the first unit's first K tile
                k_at = locate(unit_from(p, idx_cur, rec_cur), 0);
                mbar_arrive_expect_tx(bar(BAR_GF), TILE_BYTES);
                load_tile(&tm_k, sK, bar(BAR_GF), k_at);
                groups = 1;
            }
            int t = 0;                                // tiles of the units before the current one
            for (int r = 0;; ++r) {
                const int slot = r % RING;
                if (r >= RING && !(ok = wait_phase(ctl, bar(BAR_UE + slot), ((r / RING) - 1) & 1))) break;
                ring[slot].idx = idx_cur;
                ring[slot].rec = rec_cur;
                mbar_arrive(bar(BAR_UF + slot));     // release: the entry is visible to the waiters
                if (idx_cur < 0) break;
                const int idx_nxt = grab_unit(p, total_units);  // its record is read for the last group
                owe_grab = idx_nxt >= 0;
                uint4 rec_nxt = make_uint4(0u, 0u, 0u, 0u);
                bool rec_nxt_loaded = false;
                const Unit u = unit_from(p, idx_cur, rec_cur);
                const int n = max(u.n[0], u.n[1]);
                if (uq >= 1 && !(ok = wait_phase(ctl, bar(BAR_QE), (uq - 1) & 1))) break;
                const int qtok = ROWS >> p.lg;
                const int qrow = u.q_start + u.pair * 2 * qtok;
                const int qhead = u.g << p.lg;
                mbar_arrive_expect_tx(bar(BAR_QF), u.n[1] > 0 ? 2 * TILE_BYTES : TILE_BYTES);
                tma_load_3d(sQ[0], &tm_q, bar(BAR_QF), 0, qhead, qrow);
                tma_load_3d(sQ[0] + HALF_BYTES, &tm_q, bar(BAR_QF), 64, qhead, qrow);
                if (u.n[1] > 0) {
                    tma_load_3d(sQ[1], &tm_q, bar(BAR_QF), 0, qhead, qrow + qtok);
                    tma_load_3d(sQ[1] + HALF_BYTES, &tm_q, bar(BAR_QF), 64, qhead, qrow + qtok);
                }
                ++uq;
                for (int j = 0; j < n; ++j) {
                    // group gu = tile + 1: V of this tile (V stage tile & 1) and K of the tile after it
                    // (K stage gu & 1); it reuses the stages of group gu - 2
                    const int gu = t + j + 1;
                    const int sg = gu & 1;
                    if (gu >= 2 && !(ok = wait_phase(ctl, bar(BAR_GE + sg), ((gu - 2) >> 1) & 1))) break;
                    const bool k_here = j + 1 < n;
                    const bool k_next = !k_here && idx_nxt >= 0;
                    const Loc v_at = k_at;
                    if (k_here) {
                        k_at = (pref_idx == idx_cur && pref_tile == j + 1) ? pref : locate(u, j + 1);
                    } else if (k_next) {
                        if (!rec_nxt_loaded) rec_nxt = unit_record(p, idx_nxt);
                        rec_nxt_loaded = true;
                        k_at = (pref_idx == idx_nxt && pref_tile == 0) ? pref : locate(unit_from(p, idx_nxt, rec_nxt), 0);
                    }
                    mbar_arrive_expect_tx(bar(BAR_GF + sg), (k_here || k_next) ? 2 * TILE_BYTES : TILE_BYTES);
                    load_tile(&tm_v, sV + (sg ^ 1) * TILE_BYTES, bar(BAR_GF + sg), v_at);
                    if (k_here || k_next) load_tile(&tm_k, sK + sg * TILE_BYTES, bar(BAR_GF + sg), k_at);
                    ++groups;
                    // look up the next group's K tile now, while that group's stages are still in use
                    if (j + 2 < n) {
                        pref = locate(u, j + 2);
                        pref_idx = idx_cur;
                        pref_tile = j + 2;
                    } else if (j + 2 == n && idx_nxt >= 0) {
                        rec_nxt = unit_record(p, idx_nxt);
                        rec_nxt_loaded = true;
                        pref = locate(unit_from(p, idx_nxt, rec_nxt), 0);
                        pref_idx = idx_nxt;
                        pref_tile = 0;
                    }
                }
                if (!ok) break;
                t += n;
                idx_cur = idx_nxt;
                rec_cur = idx_nxt >= 0 ? rec_nxt : make_uint4(0u, 0u, 0u, 0u);
            }
            // a CTA that stopped early takes what is left of the queue, so the call still makes its
            // `total` grabs and the last of them resets the counter for the next call on the plan
            if (owe_grab)
                while (grab_unit(p, total_units) >= 0) {
                }
            if (*ctl.abort) {
                // copies already issued must land before shared memory is released
                if (uq > 0) wait_drain(bar(BAR_QF), (uq - 1) & 1);
                for (int g = max(0, groups - 2); g < groups; ++g) wait_drain(bar(BAR_GF + (g & 1)), (g >> 1) & 1);
            }
        }
        __syncwarp();
        tc_fence_before();
        __syncthreads();
    } else if (warp == MMA_WARP) {
        regs_dec<kControlRegs>();
        // ---------------------------------------------------------------- MMA
        // The whole warp runs this loop in step; each tcgen05 instruction is issued by one
        // elected lane, so descriptors and counters stay warp-uniform.
        {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(ROWS, KT, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(ROWS, D, 0, 1);
            int t = 0, uq = 0;
            int cntP[2] = {0, 0}, uact[2] = {0, 0};
            bool ok = true;
            int s_left = 0;      // S MMAs of the current unit not yet issued
            // descriptors of every operand base; a K step only advances the start-address field
            // (address >> 4 in the low 14 bits; shared addresses stay below 256 KiB, so no carry)
            const uint64_t dq0 = kmajor_desc(sQ[0]), dq1 = kmajor_desc(sQ[1]);
            const uint64_t dk0 = kmajor_desc(sK), dk1 = kmajor_desc(sK + TILE_BYTES);
            const uint64_t dv0 = vmajor_desc(sV), dv1 = vmajor_desc(sV + TILE_BYTES);
            auto issue_s = [&](int X, int st) {
                const uint64_t da = X ? dq1 : dq0;
                const uint64_t db = st ? dk1 : dk0;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t koff = ((ks >> 2) * HALF_BYTES + (ks & 3) * 32) >> 4;
                    mma_ss_warp(tmem + S_COL(X), da + koff, db + koff, idesc_qk, ks > 0 ? 1u : 0u);
                }
                mma_commit_warp(bar(BAR_SF + X));
                if (--s_left == 0) mma_commit_warp(bar(BAR_QE));   // the unit's Q tiles are no longer read
            };
            for (int r = 0; ok; ++r) {
                const int slot = r % RING;
                if (!(ok = wait_warp(ctl, bar(BAR_UF + slot), (r / RING) & 1))) break;
                const int idx = ring[slot].idx;
                const uint4 rec = ring[slot].rec;
                __syncwarp();                          // every lane has read the entry
                if (lane == 0) mbar_arrive(bar(BAR_UE + slot));
                __syncwarp();
                if (idx < 0) break;
                const Unit u = unit_from(p, idx, rec);
                const int n = max(u.n[0], u.n[1]);
                s_left = u.n[0] + u.n[1];
                if (!(ok = wait_warp(ctl, bar(BAR_QF), uq & 1))) break;
                ++uq;
                // group t holds this unit's first K; only group 0 is not waited in a previous unit
                if (t == 0 && !(ok = wait_warp(ctl, bar(BAR_GF), 0))) break;
                tc_fence_after();
                issue_s(0, t & 1);
                if (u.n[1] > 0) issue_s(1, t & 1);
                mma_commit_warp(bar(BAR_GE + (t & 1)));     // group t consumed: V(t-1) earlier, K(t) now
                for (int j = 0; j < n && ok; ++j) {
                    const int tj = t + j;
                    const int st = tj & 1;                    // V stage of this tile
                    const int sg = (tj + 1) & 1;              // its group: V(tj) and K(tj + 1)
                    const int keys_here = min(KT, u.kl - j * KT);
                    const int ksteps = (keys_here + 15) >> 4;
                    const bool s_next = j + 1 < n;            // some tile still needs S(j+1)
                    // Everything this step needs except P -- the group, and at a unit's first step the
                    // previous unit's epilogue -- is taken here, while the tensor pipe still works
                    // through the batch issued last, so after P lands only issuing remains.
                    if (!(ok = wait_warp(ctl, bar(BAR_GF + sg), ((tj + 1) >> 1) & 1))) break;
                    if (j == 0) {
#pragma unroll
                        for (int X = 0; X < 2; ++X)
                            if (ok && u.n[X] > 0 && uact[X] >= 1)
                                ok = wait_warp(ctl, bar(BAR_OE + X), (uact[X] - 1) & 1);
                        if (!ok) break;
                    }
                    if (keys_here & 15) {
                        // rows past the sequence's last key may hold anything (freed blocks are not
                        // cleared); their P is zero but 0 * NaN is NaN, so clear them
                        // (16-byte chunks spread over the warp; each row is 2 halves x 8 chunks)
                        uint8_t* vt = gbase + SM_V + st * TILE_BYTES;
                        for (int i = lane; i < (ksteps * 16 - keys_here) * 16; i += 32) {
                            const int rr = keys_here + (i >> 4);
                            *reinterpret_cast<uint4*>(vt + ((i >> 3) & 1) * HALF_BYTES + rr * 128 + (i & 7) * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                    }
                    const uint64_t dvs = st ? dv1 : dv0;
#pragma unroll
                    for (int X = 0; X < 2; ++X) {
                        if (j < u.n[X]) {
                            if (!(ok = wait_warp(ctl, bar(BAR_PF + X), cntP[X] & 1))) break;
                            ++cntP[X];
                            tc_fence_after();
                            for (int ks = 0; ks < ksteps; ++ks)
                                mma_ts_warp(tmem + O_COL(X), tmem + S_COL(X) + ks * 8, dvs + ks * (16 * 128 >> 4),
                                       idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
                            if (j == u.n[X] - 1) {
                                mma_commit_warp(bar(BAR_OF + X));
                                ++uact[X];
                            }
                        }
                        if (j + 1 < u.n[X]) {
                            tc_fence_after();
                            issue_s(X, (tj + 1) & 1);
                        }
                    }
                    if (!ok) break;
                    // the group is consumed once S(tj+1) is issued; on a unit's last tile its K belongs
                    // to the next unit, whose start commits it
                    if (s_next) mma_commit_warp(bar(BAR_GE + sg));
                }
                t += n;
            }
            mma_commit_warp(bar(BAR_DRAIN));
            wait_drain(bar(BAR_DRAIN), 0);
            __syncwarp();
        }
        __syncwarp();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    } else if (warp < 8) {
        regs_inc<kSoftmaxRegs>();
        // ---------------------------------------------------------------- softmax, tile X
        const int X = warp >> 2;                  // 0: warps 0-3, 1: warps 4-7
        const int row = tid & 127;                // TMEM lane
        const int ti = row >> p.lg;               // token of this row within the tile
        const int qtok = ROWS >> p.lg;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_tmem = tmem + lane_off + S_COL(X);
        const uint32_t o_tmem = tmem + lane_off + O_COL(X);
        const float sc = p.scale_log2;
        int cntS = 0, uact = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int slot = r % RING;
            ok = __all_sync(0xffffffffu, wait_phase(ctl, bar(BAR_UF + slot), (r / RING) & 1));
            if (!ok) break;
            const int idx = ring[slot].idx;
            const uint4 rec = ring[slot].rec;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_UE + slot));
            if (idx < 0) break;
            const Unit u = unit_from(p, idx, rec);
            const int nx = X ? u.n[1] : u.n[0];
            if (nx == 0) continue;
            const int qi = (2 * u.pair + X) * qtok + ti;
            const int jmax = min(qi + u.offset, u.kl - 1);
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < nx; ++j) {
                ok = __all_sync(0xffffffffu, wait_phase(ctl, bar(BAR_SF + X), cntS & 1));
                if (!ok) break;
                ++cntS;
                tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + 32 * c, sr[c]);
                tmem_ld_wait();
                float s[128];
#pragma unroll
                for (int e = 0; e < 128; ++e) s[e] = __uint_as_float(sr[e >> 5][e & 31]);
                const int lim = jmax - j * KT;    // columns <= lim are visible
                if (!__all_sync(0xffffffffu, lim >= KT - 1)) {
                    // the diagonal crosses this tile (or the keys end in it): hide what the row may not see
#pragma unroll
                    for (int e = 0; e < 128; ++e) s[e] = (e <= lim) ? s[e] : -INFINITY;
                }
                // row max of the raw scores (the scale is > 0), four independent 3-input chains
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int e = 0; e < 128; e += 8) {
                    mx0 = fmax3(mx0, s[e + 0], s[e + 1]);
                    mx1 = fmax3(mx1, s[e + 2], s[e + 3]);
                    mx2 = fmax3(mx2, s[e + 4], s[e + 5]);
                    mx3 = fmax3(mx3, s[e + 6], s[e + 7]);
                }
                const float m_new = fmax3(fmaxf(mx0, mx1), mx2, mx3) * sc;
                if (j == 0) {
                    m_used = m_new;
                } else if (__any_sync(0xffffffffu, m_new > m_used + kRescaleLog2)) {
                    // S_X(j) landed, so PV_X(j-1) has too: O_X is stable until P_X(j) is released
                    const float m_tgt = fmaxf(m_used, m_new);
                    const float alpha = ex2_ftz(m_used - m_tgt);
#pragma unroll 1     // a rare path, kept rolled: its registers and code stay out of the hot loop
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
                // P = 2^(s*scale - m_used) as bf16 pairs over the first 64 columns of this S buffer
                // (all of S is already in registers, so nothing is overwritten before it is read)
                const float neg_m = -m_used;
                float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int b = 32 * c + e;
                        float a0, a1, a2, a3;
                        ffma2(a0, a1, s[b], s[b + 1], sc, sc, neg_m, neg_m);
                        ffma2(a2, a3, s[b + 2], s[b + 3], sc, sc, neg_m, neg_m);
                        const float p0 = ex2_ftz(a0), p1 = ex2_ftz(a1), p2 = ex2_ftz(a2), p3 = ex2_ftz(a3);
                        fadd2(r0, r1, r0, r1, p0, p1);
                        fadd2(r2, r3, r2, r3, p2, p3);
                        pk[e >> 1] = pack_bf16x2(p0, p1);
                        pk[(e >> 1) + 1] = pack_bf16x2(p2, p3);
                    }
                    tmem_st16(s_tmem + 16 * c, pk);
                }
                l += (r0 + r1) + (r2 + r3);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(BAR_PF + X));
            }
            if (!ok) break;
            // epilogue: O_X / l -> bf16
            ok = __all_sync(0xffffffffu, wait_phase(ctl, bar(BAR_OF + X), uact & 1));
            if (!ok) break;
            ++uact;
            tc_fence_after();
            // O / l -> bf16, 64 columns at a time: each thread writes its row into this warp's
            // staging area (16-byte chunks XOR-swizzled by row, no bank conflicts), then the warp
            // stores four 128-byte row halves per instruction
            const float inv = 1.f / l;
            uint8_t* stg = gbase + SM_STAGE + warp * STAGE_WARP_BYTES;
            const uint32_t stg_s = smem_u32(stg);
#pragma unroll 1     // kept rolled: the softmax warps' code must stay small (see below)
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
                    tmem_ld32(o_tmem + 64 * half + 32 * c, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int k = 4 * c + q;                  // 16-byte chunk of the 128-byte half row
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
                        *reinterpret_cast<uint4*>(stg + lane * 128 + ((k ^ (lane & 7)) * 16)) = w;
                    }
                }
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int rr = it * 4 + (lane >> 3);          // row of this warp's 32
                    const int k = lane & 7;
                    const uint4 w = ld_shared_v4(stg_s + rr * 128 + ((k ^ (rr & 7)) * 16));
                    const int lrow = (warp & 3) * 32 + rr;        // TMEM lane = tile row
                    const int tok = (2 * u.pair + X) * qtok + (lrow >> p.lg);
                    if (tok < u.ql) {
                        uint16_t* d = p.out + (static_cast<int64_t>(u.q_start + tok) * p.num_heads + (u.g << p.lg) +
                                               (lrow & ((1 << p.lg) - 1))) * D + 64 * half + 8 * k;
                        *reinterpret_cast<uint4*>(d) = w;
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            mbar_arrive(bar(BAR_OE + X));
        }
        tc_fence_before();
        __syncthreads();
    } else {
        regs_dec<kControlRegs>();      // warps 10-11: complete the third warpgroup
        __syncthreads();
    }
}

constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t prefill_workspace_bytes(int num_seqs, int max_seqlen_q, int log_group) {
    const int unit_tok = 2 * (ROWS >> log_group);
    const size_t pairs = static_cast<size_t>(num_seqs) * ((max_seqlen_q + unit_tok - 1) / unit_tok);
    return align256((pairs + 1) * 16);
}

// The tag a plan carries: the launch arguments its records were built and checked against.
static uint32_t plan_tag(const PrefillArgs& a, int lg, int max_cost) {
    uint32_t h = 0x504b5650u;   // "PKVP"
    const uint32_t f[6] = {static_cast<uint32_t>(a.num_seqs), static_cast<uint32_t>(a.total_q),
                           static_cast<uint32_t>(lg), static_cast<uint32_t>(max_cost),
                           static_cast<uint32_t>(a.max_blocks), static_cast<uint32_t>(a.block_size)};
    for (uint32_t x : f) h = (h ^ x) * 0x01000193u;   // FNV-1a over the words
    return h;
}

pkv_status launch_prefill(const PrefillArgs& a, int* err, cudaStream_t stream, PrefillMode mode) {
    if (a.num_seqs == 0 || a.total_q == 0 || a.max_seqlen_q == 0) return PKV_OK;
    const int lg = group_log2(a.num_heads, a.num_kv_heads);
    if (lg < 0) return PKV_ERR_UNSUPPORTED;
    const int qtok = ROWS >> lg, unit_tok = 2 * qtok;
    if (a.max_seqlen_q > 0xffff * unit_tok) return PKV_ERR_UNSUPPORTED;
    const size_t need = prefill_workspace_bytes(a.num_seqs, a.max_seqlen_q, lg);
    if (a.workspace == nullptr || a.workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(a.workspace) & 15) return PKV_ERR_WORKSPACE;
    const int max_cost = 2 * ((a.max_seqlen_k + KT - 1) / KT) + 1;   // unit_cost's largest value
    const size_t plan_smem = static_cast<size_t>(max_cost + 1) * 4;
    if (plan_smem > 200 * 1024) return PKV_ERR_UNSUPPORTED;
    const uint32_t tag = plan_tag(a, lg, max_cost);

    if (!setup_once(kSetupPrefill, [] {
            return cudaFuncSetAttribute(prefill_fa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        SMEM_BYTES) == cudaSuccess &&
                   cudaFuncSetAttribute(prefill_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        200 * 1024) == cudaSuccess;
        }))
        return PKV_ERR_CUDA;
    // the setmaxnreg split inside the kernel needs this many registers per thread at launch
    static const int launch_regs = [] {
        cudaFuncAttributes fa;
        return cudaFuncGetAttributes(&fa, prefill_fa_kernel) == cudaSuccess ? fa.numRegs : -1;
    }();
    if (launch_regs < static_cast<int>(kMinLaunchRegs)) return PKV_ERR_UNSUPPORTED;

    if (mode != kPrefillRunOnly) {
        prefill_plan_kernel<<<1, 256, plan_smem, stream>>>(a.cu_q, a.cu_k, a.num_seqs, a.total_q, a.max_blocks,
                                                            a.block_size, qtok, max_cost, tag,
                                                            static_cast<uint4*>(a.workspace), err);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    }
    if (mode == kPrefillPlanOnly) return PKV_OK;

    CUtensorMap tm_q, tm_k, tm_v;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_heads),
                                  static_cast<uint64_t>(a.total_q)};
        const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.num_heads) * D * 2};
        const uint32_t box[3] = {64u, static_cast<uint32_t>(1 << lg), static_cast<uint32_t>(qtok)};
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
    p.plan = static_cast<const uint4*>(a.workspace);
    p.next_unit = static_cast<unsigned int*>(a.workspace) + 1;
    p.out = a.out;
    p.max_blocks = a.max_blocks;
    p.num_heads = a.num_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.lg = lg;
    p.block_size = a.block_size;
    p.num_blocks = a.num_blocks;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    p.tag = tag;
    p.err = err;

    const int64_t max_units = static_cast<int64_t>(a.num_seqs) *
                              ((a.max_seqlen_q + unit_tok - 1) / unit_tok) * a.num_kv_heads;
    const int grid = static_cast<int>(std::min<int64_t>(sm_count(), max_units));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, prefill_fa_kernel, tm_q, tm_k, tm_v, p) != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // namespace pkv
