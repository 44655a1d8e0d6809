// Tensor-core GEMM for the projections of the decoder (Pasos 5, 6 and 8 of "Dentro de un
// LLM: Inferencia en Python puro para Qwen3-0.6B en MLX") when a call carries more than 8
// token rows: prefill and batched decode.
//
// The product is computed transposed, D^T[m][t] = sum_k W[m][k] * H[t][k]: the weight tile
// (128 output features) is the A operand and the token tile (BN = 64/128/256 rows) the B
// operand, both K-major fp16 in shared memory with the 128-byte swizzle, fed by TMA
// (cp.async.bulk.tensor) through an mbarrier ring. One elected thread issues
// tcgen05.mma.cta_group::1.kind::f16 (M=128, N=BN, K=16, fp16 x fp16) into an fp32
// accumulator in TMEM;
// the four epilogue warps read it back with tcgen05.ld.32x32b (thread = output feature,
// registers = tokens), so every store of a token row is a coalesced 32-feature run.
// Epilogues: plain fp32 store (q|k|v), residual add into the fp32 stream (o_proj,
// down_proj), SiLU(gate) * up from two accumulators fed by the gate and up tiles (SwiGLU),
// and the LM head's per-token argmax (+ optional logits).
//
// Split-K (gridDim.z > 1, used when the tiles alone would leave most SMs idle, e.g. batched
// decode): each split accumulates a K range and writes its fp32 partial tile to a workspace;
// the CTA that finishes last for the tile (an atomic ticket, no waiting) sums the splits in
// fixed order, so results do not depend on timing, and applies the epilogue.
//
// Every mbarrier wait is bounded: after ~2 s it sets QW_DEV_TIMEOUT in the status word and
// the CTA skips the rest of its work, frees its TMEM and exits.
#include <algorithm>
#include <utility>

#include "qw_internal.h"

namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 fp16 = 128 bytes = one swizzle row
constexpr int GEMM_THREADS = 192;
constexpr unsigned long long kWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t n = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++n & 255u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitNs) return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B
// apart (SBO), descriptor version 1, start address in 16-byte units.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset
    d |= (uint64_t)1 << 46;            // version
    d |= (uint64_t)2 << 61;            // SWIZZLE_128B
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulate (bits 4-5 = 1), fp16 A and B (format
// 0 in bits 7-9 and 10-12), both K-major (bits 15, 16 clear), N >> 3 at bit 17, M >> 4 at
// bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define TMEM_LD32(taddr, r)                                                                              \
    asm volatile(                                                                                        \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15," \
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                       \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),           \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),       \
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),    \
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),    \
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])                                            \
        : "r"(taddr))

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#define TMEM_ST32(taddr, r)                                                                              \
    asm volatile(                                                                                        \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16," \
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),              \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),  \
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),      \
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),     \
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])                \
        : "memory")

template <int BN, int NA>
struct GemmCfg {
    static constexpr int A_BYTES = BM * BK * 2;  // 16 KB
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
    static constexpr int ACC_COLS = NA * BN;                 // one accumulator buffer
    static constexpr int NBUF = (2 * ACC_COLS <= 512) ? 2 : 1;
    static constexpr int TMEM_RAW = NBUF * ACC_COLS;
    static constexpr int TMEM_COLS = TMEM_RAW <= 32 ? 32 : TMEM_RAW <= 64 ? 64 : TMEM_RAW <= 128 ? 128
                                   : TMEM_RAW <= 256 ? 256 : 512;
    static constexpr int SBEST_BYTES = 4 * BN * 8;
    static constexpr int STAGES_RAW = (200 * 1024 - SBEST_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + SBEST_BYTES + 512;
};

struct GemmKParams {
    int a_row0, a2_row0, K, T, ld_out;
    int tiles_m, tiles_n, splits, units;
    float* out_f32;
    f16* out_h;
    float* logits;
    unsigned long long* best;
    int* status;
    float* part;   // split-K partial tiles [tile][split][NA*BN][128]
    int* tickets;  // split-K arrival counter per tile
};

}  // namespace

// Persistent: CTA b processes work units u = b, b + gridDim.x, ...; a unit is an output tile
// (128 features x BN tokens) and, with split-K, one K range of it. The TMA ring runs across
// units without draining; two TMEM accumulator buffers let the epilogue of one unit overlap
// the MMAs of the next. The epilogue warps hand a buffer to the MMA warp (barrier acce) only
// when it is ready for the unit that will use it: for the residual epilogue that means the
// fp32 residual tile x was loaded into it (tcgen05.st), so the MMAs compute x + W h and the
// epilogue only stores; the loads of x overlap the other buffer's MMAs.
template <int BN, int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
              const __grid_constant__ CUtensorMap tmB, GemmKParams p) {
    constexpr int NA = (EPI == EPI_SILU_MUL) ? 2 : 1;
    using C = GemmCfg<BN, NA>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned long long* sbest = reinterpret_cast<unsigned long long*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::SBEST_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* accf = bars + 2 * C::STAGES;      // [2] accumulator ready
    uint64_t* acce = bars + 2 * C::STAGES + 2;  // [2] accumulator drained
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
    volatile int* ep_fail = reinterpret_cast<volatile int*>(tmem_slot + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk_all = p.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(accf + b), 1);
            mbar_init(smem_u32(acce + b), 4);  // one arrival per epilogue warp: buffer ready
        }
        *abort_flag = 0;
        *ep_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tmA);
        if (NA == 2) tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();

    auto unit_of = [&](int u, int& tm, int& tn, int& kb0, int& kb1) {
        const int z = u % p.splits, rest = u / p.splits;
        tm = rest % p.tiles_m;
        tn = rest / p.tiles_m;
        kb0 = (nk_all * z) / p.splits;
        kb1 = (nk_all * (z + 1)) / p.splits;
    };

    if (warp == 4) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint32_t g = 0;
            for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x) {
                int tm, tn, kb0, kb1;
                unit_of(u, tm, tn, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int s = g % C::STAGES;
                    const uint32_t ph = (g / C::STAGES) & 1u;
                    if (!mbar_wait(smem_u32(empty + s), ph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        break;
                    }
                    const uint32_t st = smem_u32(smem + s * C::STAGE_BYTES);
                    mbar_expect_tx(smem_u32(full + s), C::STAGE_BYTES);
                    tma_load_2d(st, &tmA, smem_u32(full + s), kb * BK, p.a_row0 + tm * BM);
                    if (NA == 2) tma_load_2d(st + C::A_BYTES, &tmA2, smem_u32(full + s), kb * BK, p.a2_row0 + tm * BM);
                    tma_load_2d(st + NA * C::A_BYTES, &tmB, smem_u32(full + s), kb * BK, tn * BN);
                }
            }
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BM, BN);
            uint32_t g = 0;
            int i = 0;
            for (int u = blockIdx.x; u < p.units && !*abort_flag; u += gridDim.x, ++i) {
                int tm, tn, kb0, kb1;
                unit_of(u, tm, tn, kb0, kb1);
                const int buf = i % C::NBUF;
                const uint32_t use = (uint32_t)(i / C::NBUF);
                if (!mbar_wait(smem_u32(acce + buf), use & 1u, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * C::ACC_COLS;
                // the residual tile already sits in the accumulator of split 0
                const bool from_c = (EPI == EPI_RESID_F32) && (u % p.splits == 0);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int s = g % C::STAGES;
                    const uint32_t ph = (g / C::STAGES) & 1u;
                    if (!mbar_wait(smem_u32(full + s), ph, abort_flag)) {
                        ok = false;
                        *abort_flag = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + s * C::STAGE_BYTES);
                    const uint64_t ad = sw128_desc(st);
                    const uint64_t bd = sw128_desc(st + NA * C::A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint32_t acc = (kb > kb0 || k > 0 || from_c) ? 1u : 0u;
                        umma_f16(d, ad + 2 * k, bd + 2 * k, idesc, acc);
                        if (NA == 2) {
                            const uint64_t a2 = sw128_desc(st + C::A_BYTES);
                            umma_f16(d + BN, a2 + 2 * k, bd + 2 * k, idesc, acc);
                        }
                    }
                    umma_commit(smem_u32(empty + s));  // frees the stage once these MMAs finish
                }
                if (!ok) break;
                umma_commit(smem_u32(accf + buf));
            }
        }
    } else {
        // ---------------- epilogue warps 0-3: TMEM lanes 32w .. 32w+31 ----------------
        // Make buffer (i % NBUF) ready for this CTA's i-th unit and hand it to the MMA warp.
        auto prepare = [&](int i2) {
            const int u2 = blockIdx.x + i2 * gridDim.x;
            if (u2 >= p.units) return;
            const int buf2 = i2 % C::NBUF;
            if (EPI == EPI_RESID_F32 && u2 % p.splits == 0) {
                int tm2, tn2, a0, a1;
                unit_of(u2, tm2, tn2, a0, a1);
                const int n02 = tn2 * BN;
                const int f2 = tm2 * BM + warp * 32 + lane;
                const uint32_t trow2 = tmem + buf2 * C::ACC_COLS + ((uint32_t)(warp * 32) << 16);
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    uint32_t r[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = n02 + c0 + j;
                        r[j] = tok < p.T ? __float_as_uint(__ldcg(p.out_f32 + (size_t)tok * p.ld_out + f2)) : 0u;
                    }
                    TMEM_ST32(trow2 + c0, r);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(acce + buf2)) : "memory");
        };
        for (int i2 = 0; i2 < C::NBUF; ++i2) prepare(i2);
        int i = 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
            int tm, tn, kb0, kb1;
            unit_of(u, tm, tn, kb0, kb1);
            const int buf = i % C::NBUF;
            const uint32_t use = (uint32_t)(i / C::NBUF);
            // all four epilogue warps take the same decision (they meet at named barriers)
            if (!mbar_wait(smem_u32(accf + buf), use & 1u, abort_flag)) *ep_fail = 1;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const bool ok = (*ep_fail == 0);
            asm volatile("bar.sync 1, 128;" ::: "memory");
            tc_fence_after();
            if (!ok) {
                if (threadIdx.x == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
                break;
            }
            const int n0 = tn * BN;
            const int ncols = min(BN, ((p.T - n0) + 31) / 32 * 32);  // token columns holding data
            const int f = tm * BM + warp * 32 + lane;  // output feature of this thread
            const uint32_t trow = tmem + buf * C::ACC_COLS + ((uint32_t)(warp * 32) << 16);
            auto release_tmem = [&]() { prepare(i + C::NBUF); };  // this buffer's next unit
            // epilogue of 32 token columns c0.. for this thread's feature: v = accumulator,
            // u = second accumulator (up projection) for SiLU * mul
            auto apply = [&](int c0, const float* v, const float* w) {
                if (EPI == EPI_SILU_MUL) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = n0 + c0 + j;
                        if (tok < p.T) p.out_h[(size_t)tok * p.ld_out + f] = __float2half_rn(v[j] / (1.0f + expf(-v[j])) * w[j]);
                    }
                } else if (EPI == EPI_STORE_F32) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = n0 + c0 + j;
                        if (tok < p.T) p.out_f32[(size_t)tok * p.ld_out + f] = v[j];
                    }
                } else if (EPI == EPI_RESID_F32) {  // the accumulator already includes x
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = n0 + c0 + j;
                        if (tok < p.T) p.out_f32[(size_t)tok * p.ld_out + f] = v[j];
                    }
                } else {  // EPI_ARGMAX (never split)
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = n0 + c0 + j;
                        if (p.logits && tok < p.T) p.logits[(size_t)tok * p.ld_out + f] = v[j];
                        const unsigned long long key = warp_max_u64(argmax_key(v[j], f));
                        if (lane == 0) sbest[warp * BN + c0 + j] = key;
                    }
                }
            };
            if (p.splits == 1) {
                for (int c0 = 0; c0 < ncols; c0 += 32) {
                    uint32_t r[32], uu[32];
                    TMEM_LD32(trow + c0, r);
                    if (NA == 2) TMEM_LD32(trow + BN + c0, uu);
                    tmem_wait_ld();
                    if (c0 + 32 >= ncols) release_tmem();
                    float v[32], w[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        v[j] = __uint_as_float(r[j]);
                        w[j] = NA == 2 ? __uint_as_float(uu[j]) : 0.f;
                    }
                    apply(c0, v, w);
                }
                if (EPI == EPI_ARGMAX) {
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    for (int cc = threadIdx.x; cc < ncols; cc += 128) {
                        const int tok = n0 + cc;
                        if (tok < p.T) {
                            unsigned long long bb = sbest[cc];
                            for (int w2 = 1; w2 < 4; ++w2) bb = u64_max(bb, sbest[w2 * BN + cc]);
                            atomicMax(p.best + tok, bb);
                        }
                    }
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                }
            } else {
                const int z = u % p.splits;
                const int tile = tn * p.tiles_m + tm;
                float* mine = p.part + ((size_t)tile * p.splits + z) * (NA * BN) * BM;
                for (int h = 0; h < NA; ++h) {
                    for (int c0 = 0; c0 < ncols; c0 += 32) {
                        uint32_t r[32];
                        TMEM_LD32(trow + h * BN + c0, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            __stcg(mine + (size_t)(h * BN + c0 + j) * BM + warp * 32 + lane, __uint_as_float(r[j]));
                    }
                }
                release_tmem();
                __threadfence();
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (threadIdx.x == 0) *last_flag = (atomicAdd(p.tickets + tile, 1) == p.splits - 1);
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (*last_flag) {
                    __threadfence();
                    const float* base = p.part + (size_t)tile * p.splits * (NA * BN) * BM + warp * 32 + lane;
                    for (int c0 = 0; c0 < ncols; c0 += 32) {
                        float v[32], w[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = w[j] = 0.f;
                        for (int zz = 0; zz < p.splits; ++zz) {
                            const float* src = base + (size_t)zz * (NA * BN) * BM;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                v[j] += __ldcg(src + (size_t)(c0 + j) * BM);
                                if (NA == 2) w[j] += __ldcg(src + (size_t)(BN + c0 + j) * BM);
                            }
                        }
                        apply(c0, v, w);
                    }
                    if (threadIdx.x == 0) p.tickets[tile] = 0;
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");  // last_flag is reused by the next unit
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
    }
    pdl_launch();
}

namespace {

int g_gemm_sms = 0;

template <int BN, int EPI>
cudaError_t gemm_go(const LaunchCtx& c, const GemmArgs& a, int bn_idx) {
    constexpr int NA = (EPI == EPI_SILU_MUL) ? 2 : 1;
    using C = GemmCfg<BN, NA>;
    static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
    static_assert(C::STAGES >= 3, "pipeline depth");
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    GemmKParams p;
    p.a_row0 = a.a_row0;
    p.a2_row0 = a.a2_row0;
    p.K = a.K;
    p.T = a.T;
    p.ld_out = a.ld_out;
    p.out_f32 = a.out_f32;
    p.out_h = a.out_h;
    p.logits = a.logits;
    p.best = a.best;
    p.status = a.status;
    p.part = a.part;
    p.tickets = a.tickets;
    p.tiles_m = a.M / BM;
    p.tiles_n = (a.T + BN - 1) / BN;
    const int tiles = p.tiles_m * p.tiles_n;
    const int sms = a.num_sms > 0 ? a.num_sms : 148;
    int splits = 1;
    if (EPI != EPI_ARGMAX && a.part && tiles * 2 <= sms && tiles <= a.max_tiles) {
        const int nk_all = a.K / BK;
        splits = std::min(std::min(sms / tiles, 8), std::max(nk_all / 4, 1));
        while (splits > 1 && (size_t)tiles * splits * NA * BN * BM * 4 > a.part_bytes) --splits;
        splits = std::max(splits, 1);
    }
    p.splits = splits;
    p.units = tiles * splits;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(p.units, sms));
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = 0;
    if (c.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (c.counter) ++*c.counter;
    return cudaLaunchKernelEx(&cfg, k_gemm_tc<BN, EPI>, *a.tmA, *a.tmA2, a.tmB[bn_idx], p);
}

template <int EPI>
cudaError_t gemm_bn(const LaunchCtx& c, const GemmArgs& a) {
    if (a.T <= 64) return gemm_go<64, EPI>(c, a, 0);
    if (a.T <= 128 || EPI == EPI_SILU_MUL) return gemm_go<128, EPI>(c, a, 1);
    return gemm_go<256, EPI>(c, a, 2);
}

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeTiled_t get_encode() {
    static PFN_encodeTiled_t fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_encodeTiled_t)ptr;
    }
    return fn;
}

bool encode_one(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    PFN_encodeTiled_t enc = get_encode();
    if (!enc) return false;
    if (((uintptr_t)base & 15) || (cols * 2) % 16) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// box_rows == 0: encode three maps at map[0..2] with token boxes of 64, 128 and 256 rows.
bool gemm_tc_encode_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    if (box_rows) return encode_one(map, base, rows, cols, box_rows);
    return encode_one(map + 0, base, rows, cols, 64) && encode_one(map + 1, base, rows, cols, 128) &&
           encode_one(map + 2, base, rows, cols, 256);
}

cudaError_t launch_gemm_tc(const LaunchCtx& c, int epi, const GemmArgs& a) {
    if (a.M % BM || a.K % BK || a.T < 1) return cudaErrorInvalidValue;
    switch (epi) {
        case EPI_STORE_F32: return gemm_bn<EPI_STORE_F32>(c, a);
        case EPI_RESID_F32: return gemm_bn<EPI_RESID_F32>(c, a);
        case EPI_SILU_MUL: return gemm_bn<EPI_SILU_MUL>(c, a);
        case EPI_ARGMAX: return gemm_bn<EPI_ARGMAX>(c, a);
        default: return cudaErrorInvalidValue;
    }
}
