// Temperature + top-p (nucleus) sampling (Paso 8 of "Dentro de un LLM: Inferencia en Python
// puro para Qwen3-0.6B en MLX"): p = softmax(logits / T); keep the prefix of the probabilities
// in descending order (equal values by ascending token id) whose length is one more than the
// number of running sums below top_p; renormalise; draw. The draw is an inverse CDF of a given
// uniform u in [0, 1): the kept tokens are enumerated by ascending token id and the token is
// the first whose running kept probability exceeds u times the kept total. T = 0 is greedy
// argmax (lowest index on ties).
//
// k_sample_top_p: one cluster of 8 CTAs (1024 threads each) per row of logits; CTA r owns a
// contiguous eighth of the vocabulary. Nothing is sorted: the k-th largest probability that
// closes the nucleus is found by a radix select over the fp32 bit patterns of p (three
// digits of 10 bits; p >= 0, so the bit patterns order like the values): per digit, each CTA
// builds a histogram of counts and probability sums over its slice, the eight histograms are
// summed through distributed shared memory, and a suffix scan over the digits finds the one
// where the running sum from the top reaches top_p. Every probability sum is taken in fixed
// point (p * 2^40 rounded to an integer), so the sums, the nucleus and the drawn token do not
// depend on the order of the atomic additions: the result is deterministic.
#include <cstdint>

#include "qw_internal.h"

namespace {

constexpr int SP_CL = 8;           // CTAs per row (cluster)
constexpr int SP_T = 1024;         // threads per CTA
constexpr int SP_BINS = 1024;      // one radix digit (10 bits)
constexpr float SP_FIX = 1099511627776.0f;  // 2^40: fixed-point scale of probabilities

__device__ __forceinline__ uint32_t sp_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void sp_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t sp_mapa(const void* p, uint32_t rank) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(p), r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t sp_ld32(const void* p, uint32_t rank) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(sp_mapa(p, rank)) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long sp_ld64(const void* p, uint32_t rank) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(sp_mapa(p, rank)) : "memory");
    return v;
}

struct SampleP {
    const float* logits;  // [B][ld]
    size_t ld;
    int V;
    float inv_t;                  // 1 / temperature (0: greedy)
    unsigned long long tp_fix;    // top_p * 2^40
    const float* uniform;         // [B]
    int32_t* next;                // [B]
};

// One element: its probability's bit pattern (the sort key) and fixed-point value.
struct Elem {
    uint32_t key;
    unsigned long long q;
};
__device__ __forceinline__ Elem sp_elem(float l, float m, float inv_t, float inv_z) {
    const float p = expf((l - m) * inv_t) * inv_z;
    return {__float_as_uint(p), __float2ull_rn(p * SP_FIX)};
}

// Block-wide inclusive scan of one u64 per thread (1024 threads); `ws` holds 32 entries.
__device__ __forceinline__ unsigned long long sp_scan_incl(unsigned long long v, unsigned long long* ws) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) ws[w] = v;
    __syncthreads();
    if (w == 0) {
        unsigned long long s = ws[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long t = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += t;
        }
        ws[lane] = s;
    }
    __syncthreads();
    const unsigned long long r = v + (w ? ws[w - 1] : 0ull);
    __syncthreads();  // ws is reused by the next scan
    return r;
}

// Block-wide sum of one u64 per thread, returned to every thread.
__device__ __forceinline__ unsigned long long sp_sum(unsigned long long v, unsigned long long* ws) {
    const unsigned long long incl = sp_scan_incl(v, ws);
    __shared__ unsigned long long tot;
    if (threadIdx.x == SP_T - 1) tot = incl;
    __syncthreads();
    const unsigned long long r = tot;
    __syncthreads();
    return r;
}

// Add (count 1, q) to digit d of the histogram for every lane with valid d; lanes of a warp
// with the same digit are combined first (one pair of shared atomics per distinct digit).
__device__ __forceinline__ void sp_hist_add(uint32_t d, unsigned long long q, uint32_t* cnt,
                                            unsigned long long* sum) {
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    const uint32_t hi = (uint32_t)(q >> 20), lo = (uint32_t)(q & 0xFFFFFu);
    const uint32_t hs = __reduce_add_sync(peers, hi), ls = __reduce_add_sync(peers, lo);
    const int lane = threadIdx.x & 31;
    if (d < SP_BINS && lane == __ffs(peers) - 1) {
        atomicAdd(cnt + d, (uint32_t)__popc(peers));
        atomicAdd(sum + d, ((unsigned long long)hs << 20) + ls);
    }
}

}  // namespace

__global__ void __launch_bounds__(SP_T, 1) k_sample_top_p(const __grid_constant__ SampleP p) {
    __shared__ uint32_t hcnt[2][SP_BINS];            // digit histograms (two: a level is written
    __shared__ unsigned long long hsum[2][SP_BINS];  // while the previous may still be read)
    __shared__ unsigned long long ws[32];
    __shared__ unsigned long long pub64[3];          // published per-CTA totals (Z, ties, kept)
    __shared__ float pub_m;                          // published CTA max and its lowest index
    __shared__ int pub_i;
    __shared__ float wm[32];
    __shared__ int wi[32];
    __shared__ float s_m, s_inv_z;
    __shared__ int s_mi, s_digit, s_keep_all;
    __shared__ uint32_t s_cnt;
    __shared__ unsigned long long s_g, s_off;

    const int rank = (int)sp_rank(), b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int slice = (p.V + SP_CL - 1) / SP_CL;
    const int lo = min(p.V, rank * slice), hi = min(p.V, lo + slice), n = hi - lo;
    const float* row = p.logits + (size_t)b * p.ld;

    // ---- 1. the largest logit and its lowest index ------------------------------------
    float m = -INFINITY;
    int mi = 0x7fffffff;
    for (int i = lo + tid; i < hi; i += SP_T) {
        const float l = row[i];
        if (l > m) { m = l; mi = i; }  // ascending i per thread: the first maximum stays
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const int oi = __shfl_xor_sync(0xffffffffu, mi, o);
        if (om > m || (om == m && oi < mi)) { m = om; mi = oi; }
    }
    if (lane == 0) { wm[w] = m; wi[w] = mi; }
    __syncthreads();
    if (tid == 0) {
        for (int k = 1; k < 32; ++k)
            if (wm[k] > m || (wm[k] == m && wi[k] < mi)) { m = wm[k]; mi = wi[k]; }
        pub_m = m;
        pub_i = mi;
    }
    sp_cluster_sync();
    if (tid == 0) {
        float M = -INFINITY;
        int MI = 0x7fffffff;
        for (int r = 0; r < SP_CL; ++r) {
            const float rm = __uint_as_float(sp_ld32(&pub_m, r));
            const int ri = (int)sp_ld32(&pub_i, r);
            if (rm > M || (rm == M && ri < MI)) { M = rm; MI = ri; }
        }
        s_m = M;
        s_mi = MI;
    }
    __syncthreads();
    const float M = s_m;
    if (p.inv_t == 0.f) {  // greedy
        if (rank == 0 && tid == 0) p.next[b] = s_mi;
        sp_cluster_sync();  // no CTA leaves while another may read its shared memory
        return;
    }

    // ---- 2. softmax normaliser, in fixed point ----------------------------------------
    unsigned long long z = 0;
    for (int i = lo + tid; i < hi; i += SP_T) z += __float2ull_rn(expf((row[i] - M) * p.inv_t) * SP_FIX);
    z = sp_sum(z, ws);
    if (tid == 0) pub64[0] = z;
    sp_cluster_sync();
    if (tid == 0) {
        unsigned long long Z = 0;
        for (int r = 0; r < SP_CL; ++r) Z += sp_ld64(&pub64[0], r);
        s_inv_z = (float)((double)SP_FIX / (double)Z);  // p = e * 2^40 / Z
    }
    __syncthreads();
    const float inv_z = s_inv_z;

    // ---- 3. radix select of the probability that closes the nucleus --------------------
    // After level l, `prefix` holds the top 10 (l + 1) bits of that probability's key and G
    // the fixed-point sum of all probabilities with a larger key.
    uint32_t prefix = 0, tie_cnt = 0;
    unsigned long long G = 0;
    bool keep_all = false;
    for (int level = 0; level < 3 && !keep_all; ++level) {
        const int shift = 20 - 10 * level;
        uint32_t* cnt = hcnt[level & 1];
        unsigned long long* sum = hsum[level & 1];
        cnt[tid] = 0;
        sum[tid] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += SP_T) {  // the same trip count in every warp
            uint32_t d = 0xFFFFFFFFu;
            unsigned long long q = 0;
            if (base + tid < n) {
                const Elem e = sp_elem(row[lo + base + tid], M, p.inv_t, inv_z);
                if (level == 0 || (e.key >> (shift + 10)) == prefix) {
                    d = (e.key >> shift) & (SP_BINS - 1);
                    q = e.q;
                }
            }
            sp_hist_add(d, q, cnt, sum);
        }
        sp_cluster_sync();
        // thread t holds digit 1023 - t of the merged histogram: an inclusive scan gives the
        // sum over this digit and every larger one
        const int dr = SP_BINS - 1 - tid;
        uint32_t c = 0;
        unsigned long long s = 0;
        for (int r = 0; r < SP_CL; ++r) {
            c += sp_ld32(cnt + dr, r);
            s += sp_ld64(sum + dr, r);
        }
        const unsigned long long incl = sp_scan_incl(s, ws);
        if (tid == 0) s_keep_all = 0;
        __syncthreads();
        if (tid == SP_T - 1 && G + incl < p.tp_fix) s_keep_all = 1;  // rounding kept every sum below top_p
        if (G + incl >= p.tp_fix && G + incl - s < p.tp_fix) {
            s_digit = dr;
            s_g = G + incl - s;
            s_cnt = c;
        }
        __syncthreads();
        keep_all = s_keep_all != 0;
        if (!keep_all) {
            prefix = (prefix << 10) | (uint32_t)s_digit;
            G = s_g;
            tie_cnt = s_cnt;
        } else {
            G = G + incl;  // (thread 1023's value is the total; broadcast below)
        }
        __syncthreads();
    }

    // ---- 4. the kept set and its total -------------------------------------------------
    uint32_t tstar;
    unsigned long long keep_ties, S;
    if (!keep_all) {
        tstar = prefix;
        const unsigned long long qt = __float2ull_rn(__uint_as_float(tstar) * SP_FIX);
        keep_ties = qt == 0 ? tie_cnt : min((unsigned long long)tie_cnt, (p.tp_fix - G + qt - 1) / qt);
        S = G + keep_ties * qt;
    } else {
        if (tid == SP_T - 1) s_g = G;
        __syncthreads();
        S = s_g;
        tstar = 0;
        keep_ties = ~0ull;
    }

    // ---- 5. inverse-CDF draw over the kept tokens by ascending id ----------------------
    const float uf = fminf(fmaxf(p.uniform[b], 0.f), 0.99999994f);
    const unsigned long long R = min(S - 1, (unsigned long long)((double)uf * (double)S));
    const int cw = (n + SP_T - 1) / SP_T;
    const int c0 = lo + min(n, tid * cw), c1 = lo + min(n, tid * cw + cw);
    // ties below this thread's ids, cluster-wide (the nucleus keeps the lowest ids among them)
    unsigned long long tl = 0;
    for (int i = c0; i < c1; ++i) tl += sp_elem(row[i], M, p.inv_t, inv_z).key == tstar;
    const unsigned long long tincl = sp_scan_incl(tl, ws);
    if (tid == SP_T - 1) pub64[1] = tincl;
    sp_cluster_sync();
    if (tid == 0) {
        unsigned long long off = 0;
        for (int r = 0; r < rank; ++r) off += sp_ld64(&pub64[1], r);
        s_off = off;
    }
    __syncthreads();
    const unsigned long long tie0 = s_off + tincl - tl;
    __syncthreads();
    unsigned long long ks = 0, tr = tie0;
    for (int i = c0; i < c1; ++i) {
        const Elem e = sp_elem(row[i], M, p.inv_t, inv_z);
        if (e.key > tstar) {
            ks += e.q;
        } else if (e.key == tstar) {
            if (tr < keep_ties) ks += e.q;
            ++tr;
        }
    }
    const unsigned long long kincl = sp_scan_incl(ks, ws);
    if (tid == SP_T - 1) pub64[2] = kincl;
    sp_cluster_sync();
    if (tid == 0) {
        unsigned long long off = 0;
        for (int r = 0; r < rank; ++r) off += sp_ld64(&pub64[2], r);
        s_off = off;
    }
    __syncthreads();
    const unsigned long long base = s_off + kincl - ks;
    if (R >= base && R < base + ks) {  // exactly one thread of the cluster
        unsigned long long acc = base;
        tr = tie0;
        for (int i = c0; i < c1; ++i) {
            const Elem e = sp_elem(row[i], M, p.inv_t, inv_z);
            unsigned long long wq = 0;
            if (e.key > tstar) {
                wq = e.q;
            } else if (e.key == tstar) {
                if (tr < keep_ties) wq = e.q;
                ++tr;
            }
            if (R < acc + wq) {
                p.next[b] = i;
                break;
            }
            acc += wq;
        }
    }
    sp_cluster_sync();  // no CTA leaves while another may read its shared memory
}

cudaError_t launch_sample_top_p(cudaStream_t st, int B, int V, const float* logits, size_t ld, float inv_t,
                                unsigned long long tp_fix, const float* uniform, int32_t* next) {
    SampleP p;
    p.logits = logits;
    p.ld = ld;
    p.V = V;
    p.inv_t = inv_t;
    p.tp_fix = tp_fix;
    p.uniform = uniform;
    p.next = next;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(SP_CL, B);
    cfg.blockDim = dim3(SP_T);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = SP_CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_sample_top_p, p);
}
