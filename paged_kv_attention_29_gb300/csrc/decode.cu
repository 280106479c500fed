// a4: paged GQA decode attention (one query token per sequence).
//
// Visual atlas (diomchen.github.io/reference/visual-atlas.html) fig. 21: a
// decode step attends the newest token over its whole cached history; fig. 18:
// the G query heads of a group (MHA G = 1, GQA G = 2, 4, 8) read one K/V head,
// which is loaded once for all of them.  The whole step is HBM-bound (about
// 2G flops per KV byte), so the design is about keeping every SM's share of HBM
// streaming:
//
// * Teams.  A warp computes HPW = min(G, 2) query heads; a team of
//   TEAM = G / HPW warps shares one stream of staged K/V chunks, each warp
//   taking its own heads of the group.  G = 1 and G = 2 run one-warp teams.
// * Work partition.  The KV of the batch is cut into 32-token chunks, ordered
//   (sequence, KV head, chunk).  The persistent grid's W teams each take one
//   contiguous run of floor((w+1)T/W) - floor(wT/W) chunks, so every team
//   streams the same number of bytes whatever the length mix.  A step with
//   fewer than 4 chunks per team uses only ceil(T/4) teams, so short
//   sequences are not cut into single-chunk pieces that the combine must
//   then merge one round trip after another.  A run that crosses a
//   (sequence, KV head) boundary flushes a partial softmax state (running
//   max m, sum l, unnormalised o) for each piece.
// * Per-team TMA pipeline.  Each team owns TEAM x STAGES shared-memory stages
//   of one chunk of K and V (8 KiB each, 32 tokens x 256 B rows of one KV
//   head, cut out of the [num_blocks, block_size, Hkv, 128] pool by a 4-D
//   tensor map).  Lane 0 of the team's first warp keeps them all in flight; a
//   "full" mbarrier per stage tracks arrival and, for teams of more than one
//   warp, an "empty" mbarrier (one arrival per warp) frees the stage for its
//   refill.  A one-warp team refills a stage right after consuming it, with no
//   cross-warp synchronisation in the main loop.
// * Compute.  Lanes form 4 groups of 8; a group owns 8 tokens of the chunk and
//   each lane 16 of the 128 head dimensions (two 16-byte pieces, so every
//   quarter-warp shared load reads one contiguous 128-byte run: no bank
//   conflicts).  Partial dot products for both heads are reduced across the 8
//   lanes by a transposing butterfly (14 shuffles for 16 values), leaving one
//   token's score per lane; the chunk max is a warp max; the online-softmax
//   rescale of o happens once per chunk and only when the max moved.  (With
//   one head per warp the butterfly carries 8 values: 7 shuffles.)
// * Segment switches.  When a warp's run continues into the next (sequence,
//   KV head), that segment's query rows, new K/V row and length are copied
//   into the warp's shared area by cp.async as soon as the current segment
//   starts, so the switch reads shared memory instead of waiting on global
//   loads while the warp's TMA stages sit idle.
// * Combine.  A second kernel merges each (sequence, head)'s pieces in team
//   order with the log-sum-exp rule, so the result does not depend on timing.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int D = kHeadDim;
constexpr int HPW_MAX = 2;                 // query heads computed by one warp
constexpr int CHUNK = 32;                  // tokens per stage
constexpr int STAGES = 3;                  // stages per warp (a team of TEAM warps owns TEAM x STAGES)
constexpr int WARPS = 4;                   // warps per CTA (a whole number of teams of 1, 2 or 4)
constexpr int KV_TILE_BYTES = CHUNK * D * 2;
constexpr int STAGE_BYTES = 2 * KV_TILE_BYTES;
constexpr int MAX_BATCH = 4096;
constexpr int THREADS = WARPS * 32;

constexpr size_t kStageRegion = static_cast<size_t>(WARPS) * STAGES * STAGE_BYTES;
// per warp: the next segment's query rows (at most HPW_MAX), its new K and V rows, and its length
constexpr int NEXT_BYTES = HPW_MAX * D * 2 + 2 * D * 2 + 16;
constexpr size_t kNextRegion = static_cast<size_t>(WARPS) * NEXT_BYTES;

struct Params {
    const uint16_t* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int max_blocks;
    int batch;
    int num_kv_heads;
    int block_size;
    int num_blocks;
    float scale_log2;      // softmax scale * log2(e): scores live in the exp2 domain
    int total_teams;       // teams the persistent grid runs
    int32_t* plan;         // [batch + 1] chunk prefix per sequence (per KV head)
    float* part_ml;        // [pieces][G][2]  (m, l); piece = (sequence, KV head) slot + team
    float* part_o;         // [pieces][G][D]
    int* err;
    // fused KV write (pkv_decode_append): the new token of sequence b is written at
    // position context_lens[b] - 1 before the chunk holding it is loaded
    const uint16_t* k_new; // [batch, Hkv, D] or nullptr (no write)
    const uint16_t* v_new;
    uint16_t* k_pool;      // the pools the tensor maps read
    uint16_t* v_pool;
    int32_t* slot_out;     // [batch] or nullptr
};

__device__ __forceinline__ int seq_chunks(const int32_t* prefix, int b) { return prefix[b + 1] - prefix[b]; }

// Teams the run is cut over: all of them, unless that would leave fewer than KMIN chunks a
// team (a small step), where fewer, longer runs mean fewer pieces for the combine to merge.
constexpr int KMIN = 4;
__device__ __forceinline__ int run_teams(int total_teams, int64_t total) {
    const int64_t w = (total + KMIN - 1) / KMIN;
    return static_cast<int>(w < total_teams ? (w > 0 ? w : 1) : total_teams);
}

// floor(a * b / c) for non-negative operands; `narrow` (a * b known to fit in 32 bits) takes
// the unsigned 32-bit divide instead of the much longer 64-bit one.
__device__ __forceinline__ int64_t mul_div(int64_t a, int64_t b, int64_t c, bool narrow) {
    if (narrow)
        return static_cast<int64_t>(static_cast<uint32_t>(a) * static_cast<uint32_t>(b) / static_cast<uint32_t>(c));
    return a * b / c;
}

// Largest b with hkv * prefix[b] <= i  (prefix non-decreasing, prefix[0] = 0).
__device__ __forceinline__ int locate_seq(const int32_t* prefix, int batch, int hkv, int64_t i) {
    int lo = 0, hi = batch;      // invariant: hkv*prefix[lo] <= i < hkv*prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(hkv) * prefix[mid] <= i) lo = mid; else hi = mid;
    }
    return lo;
}

struct Cursor {
    int b, g, c, n;   // sequence, KV head, chunk within (b, g), chunks of b
};

__device__ __forceinline__ Cursor cursor_at(const int32_t* prefix, int batch, int hkv, int64_t i) {
    Cursor cu;
    cu.b = locate_seq(prefix, batch, hkv, i);
    cu.n = seq_chunks(prefix, cu.b);
    const int64_t rem = i - static_cast<int64_t>(hkv) * prefix[cu.b];
    cu.g = rem <= 0xffffffffll ? static_cast<int>(static_cast<uint32_t>(rem) / static_cast<uint32_t>(cu.n))
                               : static_cast<int>(rem / cu.n);
    cu.c = static_cast<int>(rem - static_cast<int64_t>(cu.g) * cu.n);
    return cu;
}

__device__ __forceinline__ void cursor_next(Cursor& cu, const int32_t* prefix, int batch, int hkv) {
    if (++cu.c < cu.n) return;
    cu.c = 0;
    if (++cu.g < hkv) return;
    cu.g = 0;
    do { ++cu.b; } while (cu.b < batch && seq_chunks(prefix, cu.b) == 0);
    cu.n = cu.b < batch ? seq_chunks(prefix, cu.b) : 0;
}

// The query rows of heads h0 .. h0 + HPW - 1 of KV head g's group (group size G).
template <int G, int HPW>
__device__ __forceinline__ void load_q(const Params& p, int b, int g, int h0, int r, float (&qf)[HPW][16]) {
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
        const uint16_t* row = p.q + (static_cast<int64_t>(b) * (p.num_kv_heads * G) + g * G + h0 + h) * D;
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(row + 8 * r));
        const uint4 c = __ldg(reinterpret_cast<const uint4*>(row + 64 + 8 * r));
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            qf[h][2 * e] = bf16_lo(w[e]) * p.scale_log2;
            qf[h][2 * e + 1] = bf16_hi(w[e]) * p.scale_log2;
        }
    }
}

// 16 dims of q . k: even and odd dims in the two halves of packed fp32x2 FMAs
// (each product rounded as a scalar fmaf would, summed in the same two chains).
__device__ __forceinline__ float dot16(const float (&qh)[16], const uint4& a, const uint4& c) {
    float s0 = 0.f, s1 = 0.f;
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) ffma2(s0, s1, qh[2 * i], qh[2 * i + 1], bf16_lo(w[i]), bf16_hi(w[i]), s0, s1);
    return s0 + s1;
}

// o += p * v over 16 dims, two dims per packed fp32x2 FMA.
__device__ __forceinline__ void axpy16(float (&oh)[16], float pw, const uint4& a, const uint4& c) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
        ffma2(oh[2 * i], oh[2 * i + 1], pw, pw, bf16_lo(w[i]), bf16_hi(w[i]), oh[2 * i], oh[2 * i + 1]);
}

// Write one piece's partial state (m, l, o) for this warp's heads h0 .. h0 + HPW - 1.
template <int G, int HPW>
__device__ __forceinline__ void flush_piece(const Params& p, int slot, int h0, int lane, const float (&m)[HPW],
                                            const float (&l)[HPW], float (&o)[HPW][16]) {
    float lsum[HPW];
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
        lsum[h] = l[h];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], off);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], 8);
            o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], 16);
        }
    }
    if (lane < 8) {
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
            float* dst = p.part_o + (static_cast<int64_t>(slot) * G + h0 + h) * D;
            float4* d0 = reinterpret_cast<float4*>(dst + 8 * lane);
            float4* d1 = reinterpret_cast<float4*>(dst + 64 + 8 * lane);
            d0[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
            d0[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
            d1[0] = make_float4(o[h][8], o[h][9], o[h][10], o[h][11]);
            d1[1] = make_float4(o[h][12], o[h][13], o[h][14], o[h][15]);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
            p.part_ml[(static_cast<int64_t>(slot) * G + h0 + h) * 2 + 0] = m[h];
            p.part_ml[(static_cast<int64_t>(slot) * G + h0 + h) * 2 + 1] = lsum[h];
        }
    }
}

// kFused: also write this step's K/V row (pkv_decode_append); a separate instantiation so
// that the plain decode compiles to the same code it had without the write.
// HPW query heads per warp, TEAM warps per team: G = HPW * TEAM.
template <bool kFused, int HPW, int TEAM>
__global__ void __launch_bounds__(THREADS, 1)
decode_splitk_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const Params p) {
    constexpr int G = HPW * TEAM;
    constexpr int NST = TEAM * STAGES;       // stages of one team
    static_assert(WARPS % TEAM == 0, "a CTA holds whole teams");
    // let the combine grid launch now; it waits for this grid's completion before reading
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // this grid may itself start while the kernel before it (typically the previous step's
    // combine) finishes: nothing global is touched before that kernel is complete
    asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1 KiB-aligned base
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStageRegion + kNextRegion);   // [WARPS * STAGES] full
    uint64_t* empty_bars = bars + WARPS * STAGES;                                     // [WARPS * STAGES] empty
    uint64_t* patch_bars = empty_bars + WARPS * STAGES;                               // [WARPS * STAGES] patched
    int32_t* prefix = reinterpret_cast<int32_t*>(patch_bars + WARPS * STAGES);
    int32_t* tsum = prefix + (p.batch + 1);
    int32_t* stage_phys = tsum + THREADS;      // [WARPS * STAGES]: physical block of each staged chunk

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int team = warp / TEAM;              // team within the CTA
    const int wt = warp - team * TEAM;         // rank within the team: heads wt*HPW .. wt*HPW + HPW - 1
    const int h0 = wt * HPW;
    const bool producer = (wt == 0);
    const int hkv = p.num_kv_heads;
    const int cap = p.max_blocks * p.block_size;

    // the block tables are read right after the prefix below: have them on their way to L2 now
    if (tid == 0) {
        uint64_t bt_bytes = static_cast<uint64_t>(p.batch) * p.max_blocks * 4;
        bt_bytes = (bt_bytes > (256u << 10) ? (256u << 10) : bt_bytes) & ~15ull;
        if ((reinterpret_cast<uintptr_t>(p.block_tables) & 15) == 0 && bt_bytes > 0)
            bulk_prefetch_l2(p.block_tables, static_cast<uint32_t>(bt_bytes));
    }

    // ---- chunk counts per sequence and their prefix (every CTA computes the same)
    const int per = (p.batch + THREADS - 1) / THREADS;
    const int b0 = tid * per;
    int local = 0;
    for (int b = b0; b < min(p.batch, b0 + per); ++b) {
        int L = __ldg(p.context_lens + b);
        if (L < 0 || L > cap) {
            if (blockIdx.x == 0) record_error(p.err, PKV_DEVERR_SEQLENS, b);
            L = L < 0 ? 0 : cap;
        }
        local += (L + CHUNK - 1) / CHUNK;
    }
    // exclusive scan of the per-thread counts: within each warp by shuffles, then over the warps
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) tsum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += tsum[w];
    const int excl = before + incl - local;
    __syncthreads();                        // every warp has read the warp totals
    tsum[tid] = excl;
    if (tid == THREADS - 1) prefix[p.batch] = excl + local;
    __syncthreads();
    {
        int run = tsum[tid];
        for (int b = b0; b < min(p.batch, b0 + per); ++b) {
            prefix[b] = run;
            int L = __ldg(p.context_lens + b);
            L = L < 0 ? 0 : (L > cap ? cap : L);
            run += (L + CHUNK - 1) / CHUNK;
        }
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int b = tid; b <= p.batch; b += THREADS) p.plan[b] = prefix[b];
    }

    // ---- this team's run of chunks (every warp of the team computes the same run)
    const int gt = blockIdx.x * (WARPS / TEAM) + team;
    const int64_t total = static_cast<int64_t>(hkv) * prefix[p.batch];
    const int W = run_teams(p.total_teams, total);
    if (gt >= W) return;
    const bool narrow = total * W <= 0xffffffffll;
    const int64_t begin = mul_div(gt, total, W, narrow);
    const int64_t end = mul_div(gt + 1, total, W, narrow);
    if (begin >= end) return;
    const int n_mine = static_cast<int>(end - begin);

    uint8_t* my_stages = smem + static_cast<size_t>(team) * NST * STAGE_BYTES;
    const uint32_t stage_base = smem_u32(my_stages);
    const uint32_t bar_base = smem_u32(bars + team * NST);
    const uint32_t empty_base = smem_u32(empty_bars + team * NST);
    const uint32_t patch_base = smem_u32(patch_bars + team * NST);
    int32_t* my_phys = stage_phys + team * NST;
    if (producer && lane == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar_base + 8 * s, 1);
            if (TEAM > 1) {
                mbar_init(empty_base + 8 * s, TEAM);
                mbar_init(patch_base + 8 * s, 1);
            }
        }
        fence_barrier_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (TEAM > 1) {
        // the other warps of the team wait on barriers the producer initialises
        asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(TEAM * 32) : "memory");
    }
    __syncwarp();
    const uint64_t policy = l2_policy_evict_first();

    // ---- producer state (first warp of the team): its own cursor and a window of 32 block-table entries
    Cursor pc = cursor_at(prefix, p.batch, hkv, begin);
    int bt_b = -1, bt_base = 0, bt_lane = -1;
    int issued = 0;
    bool failed = false;
    auto issue_next = [&]() {
        const int s = issued % NST;
        if (TEAM > 1 && issued >= NST) {
            // every warp of the team has finished with the chunk this stage held
            const bool ok = mbar_wait(empty_base + 8 * s, ((issued / NST) - 1) & 1, p.err, gt);
            if (__any_sync(0xffffffffu, !ok)) { failed = true; return; }
        }
        const int tok = pc.c * CHUNK;
        const int j = tok / p.block_size;
        if (pc.b != bt_b || j < bt_base || j >= bt_base + 32) {
            bt_b = pc.b;
            bt_base = j;
            const int jj = bt_base + lane;
            bt_lane = jj < p.max_blocks ? __ldg(p.block_tables + static_cast<int64_t>(pc.b) * p.max_blocks + jj) : -1;
        }
        const int phys = __shfl_sync(0xffffffffu, bt_lane, j - bt_base);
        if (lane == 0) {
            if (phys < 0 || phys >= p.num_blocks) record_error(p.err, PKV_DEVERR_BLOCK_ID, pc.b);
            if (kFused) my_phys[s] = phys;
            const uint32_t bar = bar_base + 8 * s;
            const uint32_t dst = stage_base + s * STAGE_BYTES;
            mbar_arrive_expect_tx(bar, STAGE_BYTES);
            const int off = tok - j * p.block_size;
            tma_load_4d_hint(dst, &tm_k, bar, 0, pc.g, off, phys, policy);
            tma_load_4d_hint(dst + KV_TILE_BYTES, &tm_v, bar, 0, pc.g, off, phys, policy);
        }
        ++issued;
        cursor_next(pc, prefix, p.batch, hkv);
    };
    if (producer) {
        const int prologue = n_mine < NST ? n_mine : NST;
        for (int i = 0; i < prologue; ++i) issue_next();
    }

    // ---- consumer (every warp of the team, each on its own heads)
    const int grp = lane >> 3;       // token group: tokens grp + 4i of the chunk
    const int r = lane & 7;          // 16 head dims: [8r, 8r+8) and [64+8r, 64+8r+8)
    Cursor cc = cursor_at(prefix, p.batch, hkv, begin);
    float qf[HPW][16], o[HPW][16], m[HPW], l[HPW];
    load_q<G, HPW>(p, cc.b, cc.g, h0, r, qf);
#pragma unroll
    for (int h = 0; h < HPW; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) o[h][e] = 0.f;
    }
    int Lb = min(max(__ldg(p.context_lens + cc.b), 0), cap);
    // fused KV write (the team's first warp): this lane's 16 bytes of the segment's new row
    // (lanes 0-15: K, 16-31: V), loaded at segment entry, used at its last chunk
    uint4 kv_row = make_uint4(0, 0, 0, 0);
    auto load_new_row = [&]() {
        if (!kFused || !producer) return;
        const int64_t src = static_cast<int64_t>(cc.b) * hkv + cc.g;
        kv_row = __ldg(reinterpret_cast<const uint4*>((lane < 16 ? p.k_new : p.v_new) + src * D + (lane & 15) * 8));
    };
    load_new_row();
    // the next segment's inputs, copied into this warp's shared area while this segment streams
    const uint32_t next_base = smem_u32(smem + kStageRegion + static_cast<size_t>(warp) * NEXT_BYTES);
    auto prefetch_next = [&](int k_at) {
        if (n_mine - k_at <= cc.n - cc.c) return;   // the run ends inside this segment
        Cursor nx = cc;
        nx.c = nx.n - 1;
        cursor_next(nx, prefix, p.batch, hkv);
        const uint16_t* qrows = p.q + (static_cast<int64_t>(nx.b) * (hkv * G) + nx.g * G + h0) * D;
        if (lane < HPW * 16)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(next_base + 16 * lane),
                         "l"(qrows + 8 * lane) : "memory");
        if (kFused && producer) {
            const int64_t src = static_cast<int64_t>(nx.b) * hkv + nx.g;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(next_base + HPW_MAX * D * 2 + 16 * lane),
                         "l"((lane < 16 ? p.k_new : p.v_new) + src * D + (lane & 15) * 8) : "memory");
        }
        if (lane == 0)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(next_base + HPW_MAX * D * 2 + 2 * D * 2),
                         "l"(p.context_lens + nx.b) : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    prefetch_next(0);
    int consumed = 0;
    // Teams of several warps: the producer patches the new row into a stage and then arrives
    // on that stage's patch barrier, which the other warps wait on.  A stage cannot be
    // patched again before every warp has released it, so each stage's barrier is at most one
    // phase ahead of any waiter; bit s holds the parity of the next phase on stage s.
    uint32_t patch_par = 0;

    for (int k = 0; k < n_mine && !failed; ++k) {
        const int s = k % NST;
        const bool ok = mbar_wait(bar_base + 8 * s, (k / NST) & 1, p.err, gt);
        if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }   // warp-uniform exit
        const uint32_t kb = stage_base + s * STAGE_BYTES;
        const uint32_t vb = kb + KV_TILE_BYTES;
        const int n_valid = min(CHUNK, Lb - cc.c * CHUNK);
        if (kFused && cc.c == cc.n - 1) {
            if (producer) {
                // the chunk holding position L - 1: put this step's K/V row of head g into the
                // staged tile (whatever the copy saw there) and into the pool, where later steps
                // read it
                const uint32_t rr = (lane < 16 ? kb : vb) + (n_valid - 1) * (D * 2) + (lane & 15) * 16;
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(rr), "r"(kv_row.x), "r"(kv_row.y),
                             "r"(kv_row.z), "r"(kv_row.w)
                             : "memory");
                const int off_in_block = (Lb - 1) % p.block_size;
                const int kv_phys = my_phys[s];   // the block the producer staged
                const bool blk_ok = kv_phys >= 0 && kv_phys < p.num_blocks;
                if (blk_ok) {
                    const int64_t row = (static_cast<int64_t>(kv_phys) * p.block_size + off_in_block) * hkv + cc.g;
                    *reinterpret_cast<uint4*>((lane < 16 ? p.k_pool : p.v_pool) + row * D + (lane & 15) * 8) = kv_row;
                }
                if (lane == 0 && cc.g == 0 && p.slot_out != nullptr)
                    p.slot_out[cc.b] = blk_ok ? kv_phys * p.block_size + off_in_block : -1;
                __syncwarp();
                // the patched row is visible to the team's other warps through the patch barrier
                if (TEAM > 1 && lane == 0) mbar_arrive(patch_base + 8 * s);
            } else if (TEAM > 1) {
                const bool pok = mbar_wait(patch_base + 8 * s, (patch_par >> s) & 1u, p.err, gt);
                if (__any_sync(0xffffffffu, !pok)) { failed = true; break; }
                patch_par ^= 1u << s;
            }
        }

        // scores: partial dot products of this lane's 16 dims, 8 tokens, HPW heads
        float part[8][HPW];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t row = kb + (grp + 4 * i) * (D * 2);
            const uint4 a = ld_shared_v4(row + 16 * r);
            const uint4 c = ld_shared_v4(row + 128 + 16 * r);
#pragma unroll
            for (int h = 0; h < HPW; ++h) part[i][h] = dot16(qf[h], a, c);
        }
        // transposing butterfly over the 8 lanes of the group: lane r ends with token grp + 4r
        float a4[4][HPW], a2[2][HPW], sc[HPW];
        const bool hA = (r & 4) != 0, hB = (r & 2) != 0, hC = (r & 1) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int h = 0; h < HPW; ++h) {
                const float send = hA ? part[j][h] : part[j + 4][h];
                const float keep = hA ? part[j + 4][h] : part[j][h];
                a4[j][h] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int h = 0; h < HPW; ++h) {
                const float send = hB ? a4[j][h] : a4[j + 2][h];
                const float keep = hB ? a4[j + 2][h] : a4[j][h];
                a2[j][h] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
            }
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
            const float send = hC ? a2[0][h] : a2[1][h];
            const float keep = hC ? a2[1][h] : a2[0][h];
            sc[h] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        }
        const bool valid = (grp + 4 * r) < n_valid;
        float pr[HPW];
        bool moved = false;
        float alpha[HPW];
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
            const float sv = valid ? sc[h] : -INFINITY;
            float cm;   // the chunk max over the warp in one reduction (no NaN reaches it: sv is a score or -inf)
            asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(cm) : "f"(sv));
            const float m_new = fmaxf(m[h], cm);
            alpha[h] = ex2_ftz(m[h] - m_new);
            moved |= (m_new != m[h]);
            m[h] = m_new;
            pr[h] = ex2_ftz(sv - m_new);
            l[h] = fmaf(l[h], alpha[h], pr[h]);
        }
        if (moved) {
#pragma unroll
            for (int h = 0; h < HPW; ++h)
#pragma unroll
                for (int e = 0; e < 16; ++e) o[h][e] *= alpha[h];
        }
        // o += p v over the group's 8 tokens
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float pw[HPW];
#pragma unroll
            for (int h = 0; h < HPW; ++h) pw[h] = __shfl_sync(0xffffffffu, pr[h], (lane & ~7) | i);
            if (grp + 4 * i < n_valid) {
                const uint32_t row = vb + (grp + 4 * i) * (D * 2);
                const uint4 a = ld_shared_v4(row + 16 * r);
                const uint4 c = ld_shared_v4(row + 128 + 16 * r);
#pragma unroll
                for (int h = 0; h < HPW; ++h) axpy16(o[h], pw[h], a, c);
            }
        }
        __syncwarp();
        ++consumed;
        if (TEAM == 1) {
            if (issued < n_mine) issue_next();        // refill the stage just consumed
        } else {
            if (lane == 0) mbar_arrive(empty_base + 8 * s);   // this warp is done with the stage
            // the producer refills the stage consumed one chunk earlier, which the other warps
            // have most likely released by now
            if (producer && k >= 1 && issued < n_mine) issue_next();
        }

        // end of this (sequence, KV head) piece or of the team's run
        if (cc.c == cc.n - 1 || k == n_mine - 1) {
            flush_piece<G, HPW>(p, cc.b * hkv + cc.g + gt, h0, lane, m, l, o);
            if (k != n_mine - 1) {
                cursor_next(cc, prefix, p.batch, hkv);
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                __syncwarp();
#pragma unroll
                for (int h = 0; h < HPW; ++h) {
                    const uint4 a = ld_shared_v4(next_base + h * D * 2 + 16 * r);
                    const uint4 c = ld_shared_v4(next_base + h * D * 2 + 128 + 16 * r);
                    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        qf[h][2 * e] = bf16_lo(w[e]) * p.scale_log2;
                        qf[h][2 * e + 1] = bf16_hi(w[e]) * p.scale_log2;
                    }
                }
                if (kFused && producer) kv_row = ld_shared_v4(next_base + HPW_MAX * D * 2 + 16 * lane);
                {
                    int len;
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(len) : "r"(next_base + HPW_MAX * D * 2 + 2 * D * 2));
                    Lb = min(max(len, 0), cap);
                }
                __syncwarp();   // every lane has read the area before the next copy lands in it
                prefetch_next(k + 1);
#pragma unroll
                for (int h = 0; h < HPW; ++h) {
                    m[h] = -INFINITY;
                    l[h] = 0.f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[h][e] = 0.f;
                }
            }
        } else {
            ++cc.c;
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (failed && producer) {
        // let the team's copies in flight land before the CTA's shared memory goes away
        for (int k = consumed; k < issued; ++k) {
            const bool ok = mbar_wait(bar_base + 8 * (k % NST), (k / NST) & 1, p.err, gt);
            if (__any_sync(0xffffffffu, !ok)) break;
        }
    }
}

// One warp per (sequence, query head): merge its pieces in team order.
template <int G>
__global__ void __launch_bounds__(128)
decode_combine_kernel(const Params p, int num_heads, uint16_t* __restrict__ out) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the next step's split-K may queue up
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the split-K grid's pieces are complete
    const int lane = threadIdx.x & 31;
    const int idx = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (idx >= p.batch * num_heads) return;
    const int b = idx / num_heads;
    const int h = idx - b * num_heads;
    const int g = h / G;
    const int hh = h - g * G;
    const int hkv = p.num_kv_heads;
    // the three plan entries in one round trip
    const int plan_b = p.plan[b], plan_b1 = p.plan[b + 1], plan_all = p.plan[p.batch];
    const int n = plan_b1 - plan_b;
    uint16_t* dst = out + static_cast<int64_t>(idx) * D + 4 * lane;
    if (n == 0) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
        if (h == 0 && lane == 0 && p.slot_out != nullptr) p.slot_out[b] = -1;   // nothing was written
        return;
    }
    const int64_t total = static_cast<int64_t>(hkv) * plan_all;
    const int64_t W = run_teams(p.total_teams, total);
    const int64_t start = static_cast<int64_t>(hkv) * plan_b + static_cast<int64_t>(g) * n;
    const int64_t last = start + n - 1;
    const bool narrow = total * W <= 0xffffffffll;
    // the team whose run holds chunk i: floor(((i + 1) W - 1) / total)
    auto team_of = [&](int64_t i) -> int {
        if (narrow)
            return static_cast<int>((static_cast<uint32_t>(i + 1) * static_cast<uint32_t>(W) - 1u) /
                                    static_cast<uint32_t>(total));
        return static_cast<int>(((i + 1) * W - 1) / total);
    };
    const int wf = team_of(start);
    const int wl = team_of(last);
    const int q = b * hkv + g;
    // when the grid has more teams than chunks, some teams between wf and wl own
    // nothing and left no piece: skip them
    auto owns_chunks = [&](int w) {
        return mul_div(w + 1, total, W, narrow) > mul_div(w, total, W, narrow);
    };
    // pieces are read four at a time, every load of a batch issued before any is used
    constexpr int BATCH = 4;
    float mj[BATCH], lj[BATCH];
    float4 vj[BATCH];
    bool own[BATCH];
    auto load_batch = [&](int w0) {
        // every slot q + w with w <= wl exists (q + wl < batch * Hkv + W), so the loads are
        // issued first; a slot of a team that owns no chunk was not written this call, and
        // its values are discarded unused
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            const int w = w0 + j;
            if (w <= wl) {
                const int64_t slot = static_cast<int64_t>(q + w) * G + hh;
                mj[j] = p.part_ml[slot * 2];
                lj[j] = p.part_ml[slot * 2 + 1];
                vj[j] = *reinterpret_cast<const float4*>(p.part_o + slot * D + 4 * lane);
            }
        }
#pragma unroll
        for (int j = 0; j < BATCH; ++j) own[j] = w0 + j <= wl && owns_chunks(w0 + j);
    };
    const bool one_batch = wl - wf < BATCH;
    float M = -INFINITY;
    if (one_batch) {
        load_batch(wf);   // the usual case: every load of the merge in one round trip
#pragma unroll
        for (int j = 0; j < BATCH; ++j)
            if (own[j]) M = fmaxf(M, mj[j]);
    } else {
        for (int w0 = wf; w0 <= wl; w0 += 32) {
            const int w = w0 + lane;
            if (w <= wl && owns_chunks(w)) M = fmaxf(M, p.part_ml[(static_cast<int64_t>(q + w) * G + hh) * 2]);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    }
    // merge in team order
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w0 = wf; w0 <= wl; w0 += BATCH) {
        if (!one_batch) load_batch(w0);
#pragma unroll
        for (int j = 0; j < BATCH; ++j) {
            if (!own[j]) continue;
            const float sc = exp2f(mj[j] - M);
            L = fmaf(sc, lj[j], L);
            acc.x = fmaf(sc, vj[j].x, acc.x);
            acc.y = fmaf(sc, vj[j].y, acc.y);
            acc.z = fmaf(sc, vj[j].z, acc.z);
            acc.w = fmaf(sc, vj[j].w, acc.w);
        }
    }
    const float inv = 1.f / L;
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(dst) = packed;
}

size_t dynamic_smem_bytes(int batch) {
    return kStageRegion + kNextRegion + 3 * WARPS * STAGES * 8 + static_cast<size_t>(batch + 1) * 4 + THREADS * 4 +
           WARPS * STAGES * 4 + 1024;
}

// Teams of a group size: one warp for G <= 2, G / 2 warps above.
constexpr int team_warps(int lg) { return lg <= 1 ? 1 : 1 << (lg - 1); }

constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

int decode_total_warps() { return sm_count() * WARPS; }

size_t decode_workspace_bytes(int batch, int num_kv_heads, int log_group, int total_warps) {
    const size_t G = static_cast<size_t>(1) << log_group;
    const size_t pieces = static_cast<size_t>(batch) * num_kv_heads + total_warps / team_warps(log_group);
    return align256(static_cast<size_t>(batch + 1) * 4) + align256(pieces * G * 2 * 4) +
           align256(pieces * G * D * 4);
}

namespace {

template <bool kFused, int HPW, int TEAM>
cudaError_t launch_splitk(const cudaLaunchConfig_t& cfg, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                          const Params& p) {
    return cudaLaunchKernelEx(&cfg, decode_splitk_kernel<kFused, HPW, TEAM>, tm_k, tm_v, p);
}

template <int HPW, int TEAM>
bool set_smem_attrs(int max_smem) {
    return cudaFuncSetAttribute(decode_splitk_kernel<false, HPW, TEAM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_smem) == cudaSuccess &&
           cudaFuncSetAttribute(decode_splitk_kernel<true, HPW, TEAM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_smem) == cudaSuccess;
}

}  // namespace

pkv_status launch_decode(const DecodeArgs& a, int* err, cudaStream_t stream) {
    if (a.batch > MAX_BATCH) return PKV_ERR_UNSUPPORTED;
    const int lg = group_log2(a.num_heads, a.num_kv_heads);
    if (lg < 0) return PKV_ERR_UNSUPPORTED;
    const int W = decode_total_warps();
    if (W <= 0) return PKV_ERR_CUDA;
    const size_t need = decode_workspace_bytes(a.batch, a.num_kv_heads, lg, W);
    if (a.workspace == nullptr || a.workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (a.batch == 0) return PKV_OK;

    CUtensorMap tm_k, tm_v;
    const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_kv_heads),
                              static_cast<uint64_t>(a.block_size), static_cast<uint64_t>(a.num_blocks)};
    const uint64_t strides[3] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(a.num_kv_heads) * D * 2,
                                 static_cast<uint64_t>(a.block_size) * a.num_kv_heads * D * 2};
    const uint32_t box[4] = {static_cast<uint32_t>(D), 1u, static_cast<uint32_t>(CHUNK), 1u};
    if (encode_tiled(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(a.k_cache), dims,
                     strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return PKV_ERR_INVALID_ARG;
    if (encode_tiled(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(a.v_cache), dims,
                     strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return PKV_ERR_INVALID_ARG;

    const int G = 1 << lg;
    const int team = team_warps(lg);
    Params p;
    p.q = a.q;
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.max_blocks = a.max_blocks;
    p.batch = a.batch;
    p.num_kv_heads = a.num_kv_heads;
    p.block_size = a.block_size;
    p.num_blocks = a.num_blocks;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    p.total_teams = W / team;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    const size_t pieces = static_cast<size_t>(a.batch) * a.num_kv_heads + p.total_teams;
    p.plan = reinterpret_cast<int32_t*>(ws);
    ws += align256(static_cast<size_t>(a.batch + 1) * 4);
    p.part_ml = reinterpret_cast<float*>(ws);
    ws += align256(pieces * G * 2 * 4);
    p.part_o = reinterpret_cast<float*>(ws);
    p.err = err;
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.k_pool = const_cast<uint16_t*>(a.k_cache);
    p.v_pool = const_cast<uint16_t*>(a.v_cache);
    p.slot_out = a.slot_out;

    const size_t smem = dynamic_smem_bytes(a.batch);
    if (!setup_once(kSetupDecode, [] {
            const int max_smem = static_cast<int>(dynamic_smem_bytes(MAX_BATCH));
            return set_smem_attrs<1, 1>(max_smem) && set_smem_attrs<2, 1>(max_smem) &&
                   set_smem_attrs<2, 2>(max_smem) && set_smem_attrs<2, 4>(max_smem);
        }))
        return PKV_ERR_CUDA;
    // both launches are programmatic dependents of what precedes them in the stream; each kernel
    // waits (griddepcontrol.wait) for its predecessor's completion before touching global memory
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(W / WARPS);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const bool fused = p.k_new != nullptr;
        cudaError_t e = cudaErrorInvalidValue;
        switch (lg) {
            case 0: e = fused ? launch_splitk<true, 1, 1>(cfg, tm_k, tm_v, p) : launch_splitk<false, 1, 1>(cfg, tm_k, tm_v, p); break;
            case 1: e = fused ? launch_splitk<true, 2, 1>(cfg, tm_k, tm_v, p) : launch_splitk<false, 2, 1>(cfg, tm_k, tm_v, p); break;
            case 2: e = fused ? launch_splitk<true, 2, 2>(cfg, tm_k, tm_v, p) : launch_splitk<false, 2, 2>(cfg, tm_k, tm_v, p); break;
            case 3: e = fused ? launch_splitk<true, 2, 4>(cfg, tm_k, tm_v, p) : launch_splitk<false, 2, 4>(cfg, tm_k, tm_v, p); break;
        }
        if (e != cudaSuccess) return PKV_ERR_CUDA;
    }
    // the combine is launched as a programmatic dependent of the split-K grid: its CTAs are
    // resident (waiting in griddepcontrol.wait) by the time the last split-K warp finishes
    const int n_rows = a.batch * a.num_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((n_rows + 3) / 4);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaErrorInvalidValue;
    switch (lg) {
        case 0: e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<1>, p, a.num_heads, a.out); break;
        case 1: e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<2>, p, a.num_heads, a.out); break;
        case 2: e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<4>, p, a.num_heads, a.out); break;
        case 3: e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<8>, p, a.num_heads, a.out); break;
    }
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // namespace pkv
