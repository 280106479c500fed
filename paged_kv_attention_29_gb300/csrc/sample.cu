// a5: temperature sampler by exponential race.
//
// Visual atlas (diomchen.github.io/reference/visual-atlas.html) fig. 23: the
// sampler's winner is argmax_v p_v / e_v with p = softmax(logits / T) and
// e_v ~ Exp(1) (equivalently argmin e_v / p_v); it is not argmax p.
//
// Because p_v = exp(logits_v / T - c) for a row constant c, the winner is
// also argmax_v (logits_v / T - ln e_v): one pass over the logits, no softmax
// normalisation.  Each row is cut into 8 slices, one per CTA of a thread-block
// cluster; a CTA reduces its slice to (best key, lowest index), and the
// cluster's first CTA merges the 8 results through distributed shared memory,
// so no global scratch or second launch is needed.
//
// Noise: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11), one call per 4
// consecutive columns: counter (column / 4, row + offset low, row + offset
// high, 0), key (seed low, seed high).  Word x of a column gives
// u = (2 (x >> 9) + 1) 2^-24, exact in fp32 and strictly inside (0, 1), and
// e = -ln u > 0.
#include <cooperative_groups.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace cg = cooperative_groups;

namespace pkv {
namespace {

constexpr int CLUSTER = 8;
constexpr int THREADS = 256;

// Philox4x32 round constants from the SC'11 paper (multipliers and Weyl increments).
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// Philox4x32-10 (ten rounds of two 32x32 -> 64 products, the high halves xored into the
// other words with the round key, which advances by the Weyl increments) for the counters
// (q, c1, c2, 0) of one row: the words that do not depend on q make round 0's second
// product and round 1's first product row constants, computed once.
struct PhiloxRow {
    uint32_t x0, y0, p_hi, p_lo, k0, k1;
};
__device__ __forceinline__ PhiloxRow philox_row(uint32_t c1, uint32_t c2, uint32_t k0, uint32_t k1) {
    PhiloxRow r;
    const uint64_t a = static_cast<uint64_t>(kPhiloxM1) * c2;
    r.x0 = static_cast<uint32_t>(a >> 32) ^ c1 ^ k0;
    r.y0 = static_cast<uint32_t>(a);
    const uint64_t p = static_cast<uint64_t>(kPhiloxM0) * r.x0;
    r.p_hi = static_cast<uint32_t>(p >> 32);
    r.p_lo = static_cast<uint32_t>(p);
    r.k0 = k0;
    r.k1 = k1;
    return r;
}
// The ten round keys of both words.  With a host seed they are computed on the host and
// read from the kernel's parameters, so the rounds spend no instruction on them.
struct RoundKeys {
    uint32_t k0[10], k1[10];
};
template <bool kParamKeys>
__device__ __forceinline__ uint32_t round_key(const RoundKeys& rk, uint32_t base, int word, int round) {
    if (kParamKeys) return word == 0 ? rk.k0[round] : rk.k1[round];
    return base + static_cast<uint32_t>(round) * (word == 0 ? kPhiloxW0 : kPhiloxW1);
}
template <bool kParamKeys>
__device__ __forceinline__ uint4 philox_row_at(uint32_t q, const PhiloxRow& r, const RoundKeys& rk) {
    const uint64_t b = static_cast<uint64_t>(kPhiloxM0) * q;            // round 0
    const uint32_t z0 = static_cast<uint32_t>(b >> 32) ^ round_key<kParamKeys>(rk, r.k1, 1, 0);
    const uint32_t w0 = static_cast<uint32_t>(b);
    const uint64_t d = static_cast<uint64_t>(kPhiloxM1) * z0;           // round 1
    uint4 c = make_uint4(static_cast<uint32_t>(d >> 32) ^ r.y0 ^ round_key<kParamKeys>(rk, r.k0, 0, 1),
                         static_cast<uint32_t>(d), r.p_hi ^ w0 ^ round_key<kParamKeys>(rk, r.k1, 1, 1), r.p_lo);
#pragma unroll
    for (int round = 2; round < 10; ++round) {
        const uint32_t k0 = round_key<kParamKeys>(rk, r.k0, 0, round);
        const uint32_t k1 = round_key<kParamKeys>(rk, r.k1, 1, round);
        const uint64_t e0 = static_cast<uint64_t>(kPhiloxM0) * c.x;
        const uint64_t e1 = static_cast<uint64_t>(kPhiloxM1) * c.z;
        c = make_uint4(static_cast<uint32_t>(e1 >> 32) ^ c.y ^ k0, static_cast<uint32_t>(e1),
                       static_cast<uint32_t>(e0 >> 32) ^ c.w ^ k1, static_cast<uint32_t>(e0));
    }
    return c;
}

// 1 - u of a noise word, exactly: with m = x >> 9, f = 1 + (2^23 - 1 - m) 2^-23 in [1, 2) has the
// complemented mantissa bits, and 1 - u = (2^24 - 2m - 1) 2^-24 = f - (1 - 2^-24), a difference
// of two floats within a factor of two of each other and therefore exact.
// ex2.approx, which the candidate bounds use, is within 2^-22 relatively, well inside their
// 1.001 margin; a bound flushed to zero only skips elements that cannot win (1 - u >= 2^-24).
__device__ __forceinline__ float one_minus_u_of(uint32_t x) {
    const float f = __uint_as_float(0x3F800000u | (~x >> 9));
    return f - 0.999999940395355224609375f;
}

// (key, index) with "better" = larger key, then lower index; index < 0 = none.
__device__ __forceinline__ bool better(float k, int i, float bk, int bi) {
    if (i < 0) return false;
    if (bi < 0) return true;
    return (k > bk) || (k == bk && i < bi);
}

__device__ __forceinline__ void consider(float logit, float inv_t, uint32_t x, int col, float& bk, int& bi) {
    // e = -ln u.  Near u = 1, where e is tiny and the key large, e must come from the exact
    // w = 1 - u (u = 1 - k 2^-24 gives e ~ k 2^-24, far below the absolute error of a fast
    // logarithm of u itself, which then mis-ranks exactly the elements most likely to win):
    // for w < 2^-6, e = -ln(1 - w) = w + w^2/2 + w^3/3 + w^4/4 + ..., the dropped terms
    // below 2^-24 of e.  Elsewhere |ln u| > 2^-6 and the hardware log2 (absolute error about
    // 1e-7) gives e to better than 1e-5 relative; the key -ln e then has an absolute error
    // below 1e-5, well inside the spacing at which two candidates could swap.
    const uint32_t m = x >> 9;
    const float w = __uint2float_rn(2u * (0x7fffffu - m) + 1u) * 5.9604644775390625e-08f;   // 1 - u, exact
    float e;
    if (w < 0.015625f) {
        e = w * fmaf(w, fmaf(w, fmaf(w, 0.25f, 0.333333343f), 0.5f), 1.0f);
    } else {
        const float u = __uint2float_rn(2u * m + 1u) * 5.9604644775390625e-08f;               // 2^-24
        e = -__logf(u);
    }
    const float key = logit * inv_t - __logf(e);
    // NaN keys never win; a -inf key only wins against nothing and is rejected
    if (key == key && key > -INFINITY && better(key, col, bk, bi)) {
        bk = key;
        bi = col;
    }
}

// kParamKeys: the seed came from the host and `rk` holds its round keys; otherwise the
// seed and row offset are read from `seed_offset` and the keys computed here.
// The loop is bound by instruction issue, so the kernel is held to 32 registers: eight
// CTAs (64 warps) resident per SM.
template <bool kParamKeys>
__global__ void __cluster_dims__(CLUSTER, 1, 1) __launch_bounds__(THREADS, 8)
sample_race_kernel(const float* __restrict__ logits, int vocab, int64_t row_stride,
                   const float* __restrict__ temperatures, uint32_t key0, uint32_t key1,
                   uint64_t offset, const uint64_t* __restrict__ seed_offset, int vec_ok,
                   int64_t* __restrict__ out_ids, int* err, const RoundKeys rk) {
    __shared__ float s_key[THREADS / 32];
    __shared__ int s_idx[THREADS / 32];
    __shared__ float c_key;
    __shared__ int c_idx;

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int row = blockIdx.y;
    const int tid = threadIdx.x;
    const float T = __ldg(temperatures + row);
    if (!kParamKeys) {                      // seed and row offset from device memory
        const uint64_t sd = __ldg(seed_offset);
        key0 = static_cast<uint32_t>(sd);
        key1 = static_cast<uint32_t>(sd >> 32);
        offset = __ldg(seed_offset + 1);
    }
    const bool t_ok = (T > 0.f) && (T < INFINITY);

    float bk = -INFINITY;
    int bi = -1;
    if (t_ok) {
        const float inv_t = 1.0f / T;
        const float inv_t_log2e = inv_t * 1.4426950408889634f;
        const uint64_t rr = static_cast<uint64_t>(row) + offset;
        const uint32_t c1 = static_cast<uint32_t>(rr);
        const uint32_t c2 = static_cast<uint32_t>(rr >> 32);
        const PhiloxRow prow = philox_row(c1, c2, key0, key1);
        const float* lrow = logits + static_cast<int64_t>(row) * row_stride;
        const int nquads = (vocab + 3) >> 2;
        const int per = (nquads + CLUSTER - 1) / CLUSTER;
        const int q0 = rank * per;
        const int q1 = min(nquads, q0 + per);
        // Pruning.  With t = best - l/T, an element can beat `best` only if
        // -ln(-ln u) > t, i.e. -ln u < e^-t; since -ln u >= 1 - u that needs
        // 1 - u < e^-t.  `best` is the warp's running maximum; t carries a 1e-3
        // margin and the bound a factor 1.001, so rounding and exact ties are
        // always decided by the exact key.  Every quad draws its noise (a test of
        // its largest logit against `best` before the Philox call -- no candidate
        // is possible when l/T + 16.7 < best, since -ln(-ln u) <= 16.64 for every
        // u the generator makes -- skips only about 6% of the calls here and cost
        // more than it saved).  A quad is first tested as a whole: its smallest
        // 1 - u (its largest word) against the bound of its largest logit.  Any
        // candidate passes that test, and only a passing quad tests its elements
        // one by one and takes the exact key of each candidate.  Skipped elements
        // cannot change the winner: some element of the warp already has a larger key.
        const int iters = (q1 - q0 + THREADS - 1) / THREADS;     // uniform across the CTA
        float wbest = -INFINITY;
        // the next quad's logits are loaded one iteration ahead, so the load is in flight while
        // this quad is examined
        auto load_quad = [&](int qd, float (&l)[4]) {
            const int col = qd * 4;
            if (qd < q1 && vec_ok && col + 3 < vocab) {
                const float4 l4 = __ldcs(reinterpret_cast<const float4*>(lrow + col));
                l[0] = l4.x; l[1] = l4.y; l[2] = l4.z; l[3] = l4.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) l[e] = (qd < q1 && col + e < vocab) ? __ldcs(lrow + col + e) : -INFINITY;
            }
        };
        auto examine = [&](int qd, const float (&l)[4]) {
            const int col = qd * 4;
            const float best = wbest;     // the warp's best after the previous quad, so never below bk
            const float lmax = fmax3(l[0], l[1], fmaxf(l[2], l[3]));
            const uint4 x = philox_row_at<kParamKeys>(static_cast<uint32_t>(qd), prow, rk);
            // candidate test: 1 - u < 1.001 e^-t, t = best - l/T - 1e-3, as 1 - u < 2^(l (log2 e / T) + cb).
            // t <= 0 gives a bound above 1 (always a candidate); l = -inf (padding past the
            // vocabulary) gives 0 (never); NaN never.
            const float cb = (1e-3f - best) * 1.4426950408889634f + 1.4419741739064e-3f;   // + log2 1.001
            const uint32_t xmax = max(max(x.x, x.y), max(x.z, x.w));
            if (one_minus_u_of(xmax) < ex2_ftz(fmaf(lmax, inv_t_log2e, cb))) {
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (one_minus_u_of(xs[e]) < ex2_ftz(fmaf(l[e], inv_t_log2e, cb)))
                        consider(l[e], inv_t, xs[e], col + e, bk, bi);
            }
        };
        // iterations in which every thread's quad exists and is four aligned columns: no checks
        const int q1_whole = (vocab & 3) ? min(q1, nquads - 1) : q1;
        const int nbulk = vec_ok ? max(0, (q1_whole - q0) / THREADS) : 0;
        float ln[4];
        load_quad(q0 + tid, ln);
        int it = 0;
        for (; it < nbulk; ++it) {
            const int qd = q0 + it * THREADS + tid;
            const float l[4] = {ln[0], ln[1], ln[2], ln[3]};
            if (it + 1 < nbulk) {
                const float4 l4 = __ldcs(reinterpret_cast<const float4*>(lrow + (qd + THREADS) * 4));
                ln[0] = l4.x; ln[1] = l4.y; ln[2] = l4.z; ln[3] = l4.w;
            } else if (it + 1 < iters) {
                load_quad(qd + THREADS, ln);
            }
            examine(qd, l);
            // share the running best across the warp (NaN never enters a key)
            asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(wbest) : "f"(bk));
        }
        for (; it < iters; ++it) {
            const int qd = q0 + it * THREADS + tid;
            const float l[4] = {ln[0], ln[1], ln[2], ln[3]};
            if (it + 1 < iters) load_quad(qd + THREADS, ln);
            if (qd < q1) examine(qd, l);
            asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(wbest) : "f"(bk));
        }
    } else if (rank == 0 && tid == 0) {
        record_error(err, PKV_DEVERR_TEMPERATURE, row);
    }
    // warp, then CTA reduction
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, bk, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ok, oi, bk, bi)) { bk = ok; bi = oi; }
    }
    if ((tid & 31) == 0) { s_key[tid >> 5] = bk; s_idx[tid >> 5] = bi; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < THREADS / 32; ++w)
            if (better(s_key[w], s_idx[w], bk, bi)) { bk = s_key[w]; bi = s_idx[w]; }
        c_key = bk;
        c_idx = bi;
    }
    // cluster reduction through distributed shared memory
    cluster.sync();
    if (rank == 0 && tid == 0) {
        float k = c_key;
        int i = c_idx;
        for (int r = 1; r < CLUSTER; ++r) {
            const float rk = *cluster.map_shared_rank(&c_key, r);
            const int ri = *cluster.map_shared_rank(&c_idx, r);
            if (better(rk, ri, k, i)) { k = rk; i = ri; }
        }
        out_ids[row] = t_ok ? static_cast<int64_t>(i) : -1;
    }
    cluster.sync();   // keep every CTA's shared memory alive until rank 0 has read it
}

}  // namespace

cudaError_t launch_sample(const float* logits, int batch, int vocab, int64_t row_stride,
                          const float* temperatures, uint64_t seed, uint64_t offset,
                          const uint64_t* seed_offset, int64_t* out_ids, int* err, cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    const int vec_ok = ((reinterpret_cast<uintptr_t>(logits) & 15) == 0) && (row_stride % 4 == 0);
    dim3 grid(CLUSTER, batch);
    RoundKeys rk = {};
    const uint32_t key0 = static_cast<uint32_t>(seed), key1 = static_cast<uint32_t>(seed >> 32);
    if (seed_offset == nullptr) {
        for (int r = 0; r < 10; ++r) {
            rk.k0[r] = key0 + static_cast<uint32_t>(r) * kPhiloxW0;
            rk.k1[r] = key1 + static_cast<uint32_t>(r) * kPhiloxW1;
        }
        sample_race_kernel<true><<<grid, THREADS, 0, stream>>>(logits, vocab, row_stride, temperatures, key0, key1,
                                                               offset, nullptr, vec_ok, out_ids, err, rk);
    } else {
        sample_race_kernel<false><<<grid, THREADS, 0, stream>>>(logits, vocab, row_stride, temperatures, key0,
                                                                key1, offset, seed_offset, vec_ok, out_ids, err, rk);
    }
    return cudaGetLastError();
}

}  // namespace pkv
