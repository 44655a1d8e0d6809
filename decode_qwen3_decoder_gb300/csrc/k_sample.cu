// Temperature + top-p (nucleus) sampling (Paso 8 of "Dentro de un LLM: Inferencia en Python
// puro para Qwen3-0.6B en MLX"): p = softmax(logits / T); keep the prefix of the probabilities
// in descending order (equal values by ascending token id) whose length is one more than the
// number of running sums below top_p; renormalise; draw. The draw is an inverse CDF of a given
// uniform u in [0, 1): the kept tokens are enumerated by ascending token id and the token is
// the first whose running kept probability exceeds u times the kept total. T = 0 is greedy
// argmax (lowest index on ties).
//
// k_sample_top_p: one cluster of 8 CTAs (1024 threads each) per row of logits; CTA r owns a
// contiguous eighth of the vocabulary and keeps the bit patterns of its probabilities in
// shared memory (p >= 0, so the bit patterns order like the values). Nothing is sorted: the
// probability that closes the nucleus is found by a radix select over those bit patterns
// (digits of 8, 8, 8 and 6 bits): per digit, each CTA sums the probabilities of its slice
// into lane-private histograms (no two lanes of a warp touch the same address), the eight
// CTAs' histograms are added through distributed shared memory, and a suffix scan over the
// digits finds the one where the running sum from the top reaches top_p. Every probability
// sum is taken in fixed point (p * 2^40 rounded to an integer), so the sums, the nucleus and
// the drawn token do not depend on the order of the atomic additions: the result is
// deterministic.
#include <cstdint>

#include "qw_internal.h"

namespace {

constexpr int SP_CL = 8;                     // CTAs per row (cluster)
constexpr int SP_T = 1024;                   // threads per CTA
constexpr int SP_BINS = 256;                 // histogram bins (digits of up to 8 bits)
constexpr int SP_HP = SP_BINS + 1;           // padded pitch of a lane's histogram (bank spread)
constexpr int SP_MAX_SLICE = 24576;          // vocabulary entries per CTA held in shared memory
constexpr float SP_FIX = 1099511627776.0f;   // 2^40: fixed-point scale of probabilities
constexpr int SP_SMEM = SP_MAX_SLICE * 4 + 32 * SP_HP * 8 + 2 * SP_BINS * 8;

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

__device__ __forceinline__ unsigned long long sp_fix(uint32_t key) {
    return __float2ull_rn(__uint_as_float(key) * SP_FIX);
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

}  // namespace


// Keys are the fp32 bit patterns of probabilities in [0, 1]: 30 significant bits, taken as
// digits of 8, 8, 8 and 6 bits (shifts 22, 14, 6, 0).
__global__ void __launch_bounds__(SP_T, 1) k_sample_top_p(const __grid_constant__ SampleP p) {
    extern __shared__ __align__(16) uint8_t sp_smem[];
    uint32_t* keys = reinterpret_cast<uint32_t*>(sp_smem);                                 // [slice]
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(sp_smem + SP_MAX_SLICE * 4);  // [32][SP_HP]
    unsigned long long* msum = hist + 32 * SP_HP;  // [2][SP_BINS] this CTA's histogram (two levels deep)
    __shared__ unsigned long long ws[32];
    __shared__ unsigned long long pub64[3];  // published per-CTA totals (Z, ties, kept)
    __shared__ float pub_m;                  // published CTA max and its lowest index
    __shared__ int pub_i;
    __shared__ float wm[32];
    __shared__ int wi[32];
    __shared__ float s_m, s_inv_z;
    __shared__ int s_mi, s_digit, s_keep_all;
    __shared__ unsigned long long s_g, s_off, s_ties;

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

    // ---- 2. exp((l - max) / T) into shared memory; the normaliser in fixed point ------
    float* ev = reinterpret_cast<float*>(keys);
    unsigned long long z = 0;
    for (int j = tid; j < n; j += SP_T) {
        const float e = expf((row[lo + j] - M) * p.inv_t);
        ev[j] = e;
        z += __float2ull_rn(e * SP_FIX);
    }
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
    for (int j = tid; j < n; j += SP_T) keys[j] = __float_as_uint(ev[j] * inv_z);
    __syncthreads();

    // ---- 3. radix select of the probability that closes the nucleus --------------------
    // After a level, `prefix` holds the key bits fixed so far and G the fixed-point sum of
    // every probability with a larger key.
    uint32_t prefix = 0;
    unsigned long long G = 0;
    bool keep_all = false;
    for (int level = 0; level < 4 && !keep_all; ++level) {
        const int bits = level == 3 ? 6 : 8, shift = level == 3 ? 0 : 22 - 8 * level, above = shift + bits;
        const uint32_t mask = (1u << bits) - 1u;
        for (int i = tid; i < 32 * SP_HP; i += SP_T) hist[i] = 0;
        __syncthreads();
        unsigned long long* mine = hist + lane * SP_HP;  // lane-private: no two lanes of a warp collide
        for (int j = tid; j < n; j += SP_T) {
            const uint32_t k = keys[j];
            if (level == 0 || (k >> above) == prefix) atomicAdd(mine + ((k >> shift) & mask), sp_fix(k));
        }
        __syncthreads();
        unsigned long long* ms = msum + (level & 1) * SP_BINS;
        if (tid < SP_BINS) {
            unsigned long long t = 0;
            for (int l = 0; l < 32; ++l) t += hist[l * SP_HP + tid];
            ms[tid] = t;
        }
        sp_cluster_sync();
        // thread t < 256 holds digit 255 - t of the cluster's histogram; the inclusive scan
        // gives the sum over that digit and every larger one
        const int dr = SP_BINS - 1 - tid;
        unsigned long long s = 0;
        if (tid < SP_BINS)
            for (int r = 0; r < SP_CL; ++r) s += sp_ld64(ms + dr, r);
        const unsigned long long incl = sp_scan_incl(s, ws);
        if (tid == 0) s_keep_all = 0;
        __syncthreads();
        if (tid == SP_T - 1 && G + incl < p.tp_fix) {  // rounding kept every running sum below top_p
            s_keep_all = 1;
            s_g = G + incl;
        }
        if (tid < SP_BINS && G + incl >= p.tp_fix && G + incl - s < p.tp_fix) {
            s_digit = dr;
            s_g = G + incl - s;
        }
        __syncthreads();
        keep_all = s_keep_all != 0;
        G = s_g;
        if (!keep_all) prefix = (prefix << bits) | (uint32_t)s_digit;
        __syncthreads();
    }

    // ---- 4. ties at the closing value (the nucleus keeps the lowest ids among them) ----
    const uint32_t tstar = keep_all ? 0u : prefix;
    const int cw = (n + SP_T - 1) / SP_T, j0 = min(n, tid * cw), j1 = min(n, j0 + cw);
    unsigned long long tl = 0;
    for (int j = j0; j < j1; ++j) tl += keys[j] == tstar;
    const unsigned long long tincl = sp_scan_incl(tl, ws);
    if (tid == SP_T - 1) pub64[1] = tincl;
    sp_cluster_sync();
    if (tid == 0) {
        unsigned long long off = 0, all = 0;
        for (int r = 0; r < SP_CL; ++r) {
            const unsigned long long v = sp_ld64(&pub64[1], r);
            if (r < rank) off += v;
            all += v;
        }
        s_off = off;
        s_ties = all;
    }
    __syncthreads();
    const unsigned long long tie0 = s_off + tincl - tl;
    unsigned long long keep_ties, S;
    if (!keep_all) {
        const unsigned long long qt = sp_fix(tstar), c = s_ties;
        keep_ties = qt == 0 ? c : min(c, (p.tp_fix - G + qt - 1) / qt);
        S = G + keep_ties * qt;
    } else {
        keep_ties = ~0ull;
        S = G;  // every token is kept: G is the total
    }
    __syncthreads();

    // ---- 5. inverse-CDF draw over the kept tokens by ascending id ----------------------
    const float uf = fminf(fmaxf(p.uniform[b], 0.f), 0.99999994f);
    const unsigned long long R = min(S - 1, (unsigned long long)((double)uf * (double)S));
    unsigned long long ks = 0, tr = tie0;
    for (int j = j0; j < j1; ++j) {
        const uint32_t k = keys[j];
        if (k > tstar) {
            ks += sp_fix(k);
        } else if (k == tstar) {
            if (tr < keep_ties) ks += sp_fix(k);
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
        for (int j = j0; j < j1; ++j) {
            const uint32_t k = keys[j];
            unsigned long long wq = 0;
            if (k > tstar) {
                wq = sp_fix(k);
            } else if (k == tstar) {
                if (tr < keep_ties) wq = sp_fix(k);
                ++tr;
            }
            if (R < acc + wq) {
                p.next[b] = lo + j;
                break;
            }
            acc += wq;
        }
    }
    sp_cluster_sync();  // no CTA leaves while another may read its shared memory
}

int sample_max_vocab() { return SP_CL * SP_MAX_SLICE; }

cudaError_t launch_sample_top_p(cudaStream_t st, int B, int V, const float* logits, size_t ld, float inv_t,
                                unsigned long long tp_fix, const float* uniform, int32_t* next) {
    if (V > SP_CL * SP_MAX_SLICE) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_sample_top_p, cudaFuncAttributeMaxDynamicSharedMemorySize, SP_SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
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
    cfg.dynamicSmemBytes = SP_SMEM;
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
