// Tensor-core GEMM for the projections of the decoder (Pasos 5, 6 and 8 of "Dentro de un
// LLM: Inferencia en Python puro para Qwen3-0.6B en MLX") when a call carries more than 8
// token rows: prefill and batched decode.
//
// The product is computed transposed, D^T[m][t] = sum_k W[m][k] * H[t][k]: the weight tile
// (128 output rows) is the A operand and the token tile (BN = 64/128/256 rows) the B
// operand, both K-major fp16 in shared memory with the 128-byte swizzle, fed by TMA
// (cp.async.bulk.tensor) through an mbarrier ring. One elected thread issues
// tcgen05.mma.cta_group::1.kind::f16 (M=128, N=BN, K=16, fp16 x fp16) into an fp32
// accumulator in TMEM; the four epilogue warps read it back with tcgen05.ld.32x32b
// (thread = output row, registers = tokens).
//
// Epilogues:
//   EPI_QKV_HEADS  one 128-row tile of the q|k|v projection is exactly one head: the tile
//                  is staged through shared memory as fp16 [token][128] and each token's head
//                  gets the per-head RMSNorm and the rotate-half RoPE (q and k heads, Pasos 4
//                  and 5), then q is stored as fp16 [T][n_heads][128] and k / v are appended
//                  (fp16) at the token's page slot of the KV cache.
//   EPI_RESID_F32  x = x + W h (o_proj, down_proj): the residual rows of the next 32 tokens
//                  are loaded while the current ones are added and stored.
//   EPI_SILU_MUL   gate and up rows are packed interleaved, 64 gate rows then the same 64 up
//                  rows per tile, so one M=128 MMA yields both; the epilogue stores
//                  SiLU(gate) * up as fp16 (Paso 6).
//   EPI_ARGMAX     the tied LM head: per-token packed argmax keys (+ optional logits).
//
// Two kernels share this machinery:
//   k_gemm_tc  persistent (one CTA per SM walks the output tiles; the TMA ring runs across
//              tiles; two TMEM accumulators let one tile's epilogue overlap the next tile's
//              MMAs). Used when the tiles fill the GPU (prefill, LM head).
//   k_gemm_cl  split-K over a thread-block cluster, one tile per cluster (batched decode,
//              where a layer has too few tiles to occupy the SMs): CTA z of the cluster
//              accumulates K range z, writes its fp32 partial for the token columns owned by
//              CTA o straight into o's shared memory (distributed shared memory), and each
//              CTA sums the partials of its own columns and applies the epilogue. Only the
//              two cluster barriers order it; nothing goes through global memory.
//
// Programmatic dependent launch: weights never change during a step, so the producer
// issues the weight tiles of the first ring stages before waiting for the previous kernel
// (griddepcontrol.wait); activations, residuals and outputs are touched only after it.
//
// Every mbarrier wait is bounded: after ~2 s it sets QW_DEV_TIMEOUT in the status word and
// the CTA skips the rest of its work, frees its TMEM and exits.
#include <algorithm>
#include <utility>

#include "qw_internal.h"
#include "tc_sm103.cuh"

#include "gemm_epi.cuh"

// =======================================================================================
// Persistent kernel: CTA b processes tiles u = b, b + gridDim.x, ...
// PAIR: clusters of two CTAs on a pair of SMs process 256-row tiles with the CTA-pair MMA
// (tcgen05.mma.cta_group::2, M = 256): CTA rank r holds weight rows [128 r, 128 r + 128) and
// token rows [r BN / 2, (r + 1) BN / 2) of each stage, so each SM loads and keeps half of the
// token tile; the leader (rank 0) issues the MMAs into both CTAs' tensor memory, and each
// CTA's epilogue reads its own 128 rows. The leader's stage barriers count both CTAs' copies;
// its MMA completions are multicast to both CTAs; the peer's epilogue frees accumulators by
// arriving on the leader's barriers.
// =======================================================================================
template <int BN, int EPI, bool PAIR>
__global__ void __launch_bounds__(GEMM_TC_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmKParams p) {
    using C = GemmCfg<BN, EPI, 2, PAIR ? 2 : 1>;
    static_assert(C::NBUF == 2, "one accumulator buffer per epilogue warpgroup");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* extra = smem + C::STAGES * C::STAGE_BYTES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = (warp < 8) ? (warp >> 2) : 0;  // epilogue warpgroup of this thread
    unsigned long long* sbest = reinterpret_cast<unsigned long long*>(extra + wg * C::SBEST_WG);
    float* E = reinterpret_cast<float*>(extra + C::SBEST_BYTES + wg * C::E_WG);
    float* nws = reinterpret_cast<float*>(extra + C::SBEST_BYTES + C::STAGE_E_BYTES);
    int* tpos = reinterpret_cast<int*>(extra + C::SBEST_BYTES + C::STAGE_E_BYTES + C::NW_BYTES + wg * C::META_WG);
    int* tdst = tpos + BN;
    uint64_t* bars = reinterpret_cast<uint64_t*>(extra + C::EXTRA);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* accf = bars + 2 * C::STAGES;      // [2] accumulator ready (buffer b: warpgroup b)
    uint64_t* acce = bars + 2 * C::STAGES + 2;  // [2] accumulator free
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* ep_fail = reinterpret_cast<volatile int*>(tmem_slot + 2) + wg;  // [2]

    const int nk = p.K / BK;
    const int rank = PAIR ? (int)cluster_rank() : 0;
    const int pid = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // CTA (pair) index
    const int npid = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int tiles_mp = PAIR ? p.tiles_m / 2 : p.tiles_m;  // tile rows of 256 (pair) or 128
    // stage barriers the copies complete on: the leader's for a pair
    auto full_bar = [&](int s) -> uint32_t {
        return PAIR ? mapa_shared(smem_u32(full + s), 0u) : smem_u32(full + s);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(accf + b), 1);
            mbar_init(smem_u32(acce + b), PAIR ? 16 : 8);  // one arrival per epilogue warp (of both CTAs)
        }
        *abort_flag = 0;
        ep_fail[0] = 0;
        ep_fail[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 9) {
        if (PAIR) {  // one warp of each CTA of the pair, collectively
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                         "r"(C::TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                         "r"(C::TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    if (EPI == EPI_QKV_HEADS && threadIdx.x < 128) load_norm_weights(p, nws);  // weights: before the wait
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();  // the peer's copies signal the leader's barriers: both initialised
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch();

    // tm: 128-row weight tile of this CTA; tn: token tile
    auto tile_of = [&](int u, int& tm, int& tn) {
        tm = PAIR ? 2 * (u % tiles_mp) + rank : u % tiles_mp;
        tn = u / tiles_mp;
    };
    const int b_off = PAIR ? rank * (BN / 2) : 0;  // this CTA's token rows within a tile

    if (warp == 8) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            // weight tiles of the first ring stages before the dependency wait
            // the leader's stage barrier expects the bytes of both CTAs' copies
            constexpr uint32_t kStageTx = (PAIR ? 2 : 1) * C::STAGE_BYTES;
            auto load = [&](uint32_t dst, const CUtensorMap* map, int s, int x, int y) {
                if (PAIR)
                    tma_load_2d_pair(dst, map, full_bar(s), x, y);
                else
                    tma_load_2d(dst, map, full_bar(s), x, y);
            };
            int pre = 0;
            {
                int u = pid, kb = 0;
                while (pre < C::STAGES && u < p.units) {
                    int tm, tn;
                    tile_of(u, tm, tn);
                    const uint32_t st = smem_u32(smem + pre * C::STAGE_BYTES);
                    if (rank == 0) mbar_expect_tx(smem_u32(full + pre), kStageTx);
                    load(st, &tmA, pre, kb * BK, p.a_row0 + tm * BM);
                    ++pre;
                    if (++kb == nk) {
                        kb = 0;
                        u += npid;
                    }
                }
            }
            pdl_wait();
            uint32_t g = 0;
            for (int u = pid; u < p.units && !*abort_flag; u += npid) {
                int tm, tn;
                tile_of(u, tm, tn);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = g % C::STAGES;
                    const uint32_t st = smem_u32(smem + s * C::STAGE_BYTES);
                    if ((int)g < pre) {  // weights already in flight
                        load(st + C::A_BYTES, &tmB, s, kb * BK, p.b_row0 + tn * BN + b_off);
                        continue;
                    }
                    const uint32_t ph = (g / C::STAGES) & 1u;
                    if (!mbar_wait(smem_u32(empty + s), ph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        break;
                    }
                    if (rank == 0) mbar_expect_tx(smem_u32(full + s), kStageTx);
                    load(st, &tmA, s, kb * BK, p.a_row0 + tm * BM);
                    load(st + C::A_BYTES, &tmB, s, kb * BK, p.b_row0 + tn * BN + b_off);
                }
            }
        }
    } else if (warp == 9) {
        // ---------------- MMA issuer (the leader of a pair) ----------------
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_f16(PAIR ? 2 * BM : BM, BN);
            uint32_t g = 0;
            int i = 0;
            for (int u = pid; u < p.units && !*abort_flag; u += npid, ++i) {
                const int buf = i % C::NBUF;
                const uint32_t use = (uint32_t)(i / C::NBUF);
                if (!mbar_wait(smem_u32(acce + buf), use & 1u, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * BN;
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb, ++g) {
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
                    const uint64_t bd = sw128_desc(st + C::A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        if (PAIR)
                            umma_f16_pair(d, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                        else
                            umma_f16(d, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    // frees the stage (in both CTAs of a pair) once these MMAs finish
                    if (PAIR)
                        umma_commit_pair(smem_u32(empty + s));
                    else
                        umma_commit(smem_u32(empty + s));
                }
                if (!ok) break;
                if (PAIR)
                    umma_commit_pair(smem_u32(accf + buf));
                else
                    umma_commit(smem_u32(accf + buf));
            }
        }
    } else {
        // ---------------- epilogue warpgroups: warp w reads TMEM lanes 32 (w % 4) .. ----------
        // both warpgroups take every tile, warpgroup wg its token columns [wg BN / 2, (wg + 1)
        // BN / 2): a tile's accumulator is read in half the time, so it is back with the MMA
        // warp well within the next tile's MMAs
        const int ew = warp & 3;  // warp within the warpgroup
        // hand buffer (i2 % NBUF) to the MMA warp for this CTA's i2-th tile
        auto prepare = [&](int i2) {
            const int u2 = pid + i2 * npid;
            if (u2 >= p.units) return;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                const uint32_t bar = smem_u32(acce + (i2 % C::NBUF));
                if (PAIR)  // the leader's MMA waits for both CTAs' epilogues
                    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mapa_shared(bar, 0u))
                                 : "memory");
                else
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
            }
        };
        prepare(0);  // both buffers start free: nothing to read, before the wait
        prepare(1);
        pdl_wait();
        int i = 0;
        const int c_lo = wg * (BN / 2);  // this warpgroup's first token column of a tile
        for (int u = pid; u < p.units; u += npid, ++i) {
            int tm, tn;
            tile_of(u, tm, tn);
            const int buf = i % C::NBUF;
            const uint32_t use = (uint32_t)(i / C::NBUF);
            if (EPI == EPI_QKV_HEADS) fill_tok_meta<BN>(p, tn * BN, tm, tpos, tdst);  // overlaps the MMAs
            float xr[32];  // EPI_RESID_F32: residual rows of the current 32 tokens
            if (EPI == EPI_RESID_F32) load_resid(p, tn * BN + c_lo, tm * BM + ew * 32 + lane, xr);
            // all four epilogue warps take the same decision (they meet at named barriers)
            if (!mbar_wait(smem_u32(accf + buf), use & 1u, abort_flag)) *ep_fail = 1;
            named_bar_epi();
            const bool ok = (*ep_fail == 0);
            named_bar_epi();
            tc_fence_after();
            if (!ok) {
                if (epi_tid() == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
                break;
            }
            const int n0 = tn * BN;
            const int ncols = min(BN, ((p.T - n0) + 31) / 32 * 32);  // token columns holding data
            const int c_hi = min(c_lo + BN / 2, ncols);                // this warpgroup's columns end
            const int fl = ew * 32 + lane;                             // tile row of this thread
            const uint32_t trow = tmem + buf * BN + ((uint32_t)(ew * 32) << 16);
            const bool rope = (EPI == EPI_QKV_HEADS) && tm < p.n_heads + p.n_kv;
            // gate/up (K = 1024: one tile of MMA time per epilogue): the next chunk's columns are
            // read from tensor memory while this chunk is processed, and the accumulator is
            // freed as soon as its last columns have landed in registers. q|k|v instead requests
            // the next chunk's RoPE rows (L2-resident table) one chunk ahead (registers allow
            // one of the two).
            constexpr bool kPipe = (EPI == EPI_SILU_MUL);
            uint32_t rnext[kPipe ? 32 : 1];
            RopeRegs rrnext;
            if (c_hi <= c_lo) prepare(i + 2);  // no columns of this tile here: free it at once
            if (kPipe && c_lo < c_hi) {
                TMEM_LD32(trow + c_lo, rnext);
                tmem_wait_ld();
                if (c_hi - c_lo <= 32) prepare(i + 2);
            }
            if (rope && c_lo < c_hi) load_rope(p, tpos, c_lo, min(32, p.T - (n0 + c_lo)), rrnext);
            for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
                uint32_t r[32];
                RopeRegs rr;  // this chunk's RoPE rows
                if (rope) {
                    rr = rrnext;
                    if (c0 + 32 < c_hi) load_rope(p, tpos, c0 + 32, min(32, p.T - (n0 + c0 + 32)), rrnext);
                }
                if (kPipe) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = rnext[j];
                    if (c0 + 32 < c_hi) TMEM_LD32(trow + c0 + 32, rnext);
                } else {
                    TMEM_LD32(trow + c0, r);
                    tmem_wait_ld();
                    if (c0 + 32 >= c_hi) prepare(i + 2);  // this buffer's next tile
                }
                if (EPI == EPI_QKV_HEADS || EPI == EPI_SILU_MUL) {
                    if (EPI == EPI_QKV_HEADS) {
                        f16* EH = reinterpret_cast<f16*>(E);
#pragma unroll
                        for (int j = 0; j < 32; ++j) EH[j * EPH + fl] = __float2half_rn(__uint_as_float(r[j]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) E[j * EP + fl] = __uint_as_float(r[j]);
                    }
                    named_bar_epi();
                    const int ntok = min(32, p.T - (n0 + c0));
                    if (EPI == EPI_QKV_HEADS) {
                        epi_heads(p, reinterpret_cast<const f16*>(E), nws, tdst, rr, n0 + c0, c0, ntok, tm);
                    } else {
                        epi_silu(p, E, n0 + c0, ntok, tm);
                    }
                    if (kPipe && c0 + 32 < c_hi) {
                        tmem_wait_ld();
                        if (c0 + 64 >= c_hi) prepare(i + 2);  // all columns read: this buffer's next tile
                    }
                    named_bar_epi();  // E is refilled by the next chunk
                } else if (EPI == EPI_RESID_F32) {
                    const int f = tm * BM + fl;
                    float xn[32];
                    if (c0 + 32 < c_hi) load_resid(p, n0 + c0 + 32, f, xn);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = n0 + c0 + j;
                        if (tok < p.T) p.out_f32[(size_t)tok * p.ld_out + f] = __uint_as_float(r[j]) + xr[j];
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) xr[j] = xn[j];
                } else {  // EPI_ARGMAX
                    const int f = tm * BM + fl;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = n0 + c0 + j;
                        const float v = __uint_as_float(r[j]);
                        if (p.logits && tok < p.T) p.logits[(size_t)tok * p.ld_out + f] = v;
                        const unsigned long long key = warp_max_u64(argmax_key(v, f));
                        if (lane == 0) sbest[ew * BN + c0 + j] = key;
                    }
                }
            }
            if (EPI == EPI_ARGMAX) {
                named_bar_epi();
                for (int cc = c_lo + epi_tid(); cc < c_hi; cc += 128) {
                    const int tok = n0 + cc;
                    if (tok < p.T) {
                        unsigned long long bb = sbest[cc];
                        for (int w2 = 1; w2 < 4; ++w2) bb = u64_max(bb, sbest[w2 * BN + cc]);
                        atomicMax(p.best + tok, bb);
                    }
                }
                named_bar_epi();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
    if (PAIR) cluster_sync_all();  // no copy, MMA or arrival of the pair still targets this CTA
    if (warp == 9) {
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                         : "memory");
    }
}

// =======================================================================================
// Cluster split-K kernel: cluster c = one output tile, CTA rank z = K range z.
// =======================================================================================
template <int BN, int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm_cl(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmKParams p) {
    using C = GemmCfg<BN, EPI, 1>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* extra = smem + C::STAGES * C::STAGE_BYTES;
    float* E = reinterpret_cast<float*>(extra + C::SBEST_BYTES);
    float* nws = reinterpret_cast<float*>(extra + C::SBEST_BYTES + C::STAGE_E_BYTES);
    int* tpos = reinterpret_cast<int*>(extra + C::SBEST_BYTES + C::STAGE_E_BYTES + C::NW_BYTES);
    int* tdst = tpos + BN;
    uint64_t* bars = reinterpret_cast<uint64_t*>(extra + C::EXTRA);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* accf = bars + 2 * C::STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* ep_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);
    // partial sums received from the cluster: [split][owned column][128 rows] fp32, over the
    // stage ring (free once every CTA of the cluster has finished its MMAs)
    float* red = reinterpret_cast<float*>(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.splits;
    const int z = (int)cluster_rank();
    const int tile = (int)cluster_id_x();
    const int tm = tile % p.tiles_m, tn = tile / p.tiles_m;
    const int nk_all = p.K / BK;
    const int kb0 = (nk_all * z) / S, kb1 = (nk_all * (z + 1)) / S;
    const int nk = kb1 - kb0;
    const int WMAX = (BN + S - 1) / S;
    const int n0 = tn * BN;
    float xr0[32];  // EPI_RESID_F32: residual rows of the first 32 owned columns (epilogue warps)

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), 1);
        }
        mbar_init(smem_u32(accf), 1);
        *abort_flag = 0;
        *ep_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tmA);
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
    pdl_launch();

    if (warp == 4) {
        if (lane == 0) {
            const int pre = min(nk, C::STAGES);
            for (int j = 0; j < pre; ++j) {  // weights first: they do not depend on the previous kernel
                mbar_expect_tx(smem_u32(full + j), C::STAGE_BYTES);
                tma_load_2d(smem_u32(smem + j * C::STAGE_BYTES), &tmA, smem_u32(full + j), (kb0 + j) * BK,
                            p.a_row0 + tm * BM);
            }
            pdl_wait();
            for (int j = 0; j < pre; ++j)
                tma_load_2d(smem_u32(smem + j * C::STAGE_BYTES) + C::A_BYTES, &tmB, smem_u32(full + j), (kb0 + j) * BK,
                            p.b_row0 + n0);
            for (int j = pre; j < nk; ++j) {
                const int s = j % C::STAGES;
                const uint32_t ph = (j / C::STAGES) & 1u;
                if (!mbar_wait(smem_u32(empty + s), ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                const uint32_t st = smem_u32(smem + s * C::STAGE_BYTES);
                mbar_expect_tx(smem_u32(full + s), C::STAGE_BYTES);
                tma_load_2d(st, &tmA, smem_u32(full + s), (kb0 + j) * BK, p.a_row0 + tm * BM);
                tma_load_2d(st + C::A_BYTES, &tmB, smem_u32(full + s), (kb0 + j) * BK, p.b_row0 + n0);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BM, BN);
            bool ok = true;
            for (int j = 0; j < nk && ok; ++j) {
                const int s = j % C::STAGES;
                const uint32_t ph = (j / C::STAGES) & 1u;
                if (!mbar_wait(smem_u32(full + s), ph, abort_flag)) {
                    ok = false;
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t st = smem_u32(smem + s * C::STAGE_BYTES);
                const uint64_t ad = sw128_desc(st);
                const uint64_t bd = sw128_desc(st + C::A_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_f16(tmem, ad + 2 * k, bd + 2 * k, idesc, (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(smem_u32(empty + s));
            }
            if (ok) umma_commit(smem_u32(accf));
        }
        __syncwarp();
    } else {
        if (EPI == EPI_QKV_HEADS) load_norm_weights(p, nws);
        pdl_wait();
        if (EPI == EPI_QKV_HEADS) fill_tok_meta<BN>(p, n0, tm, tpos, tdst);
        const int fl = warp * 32 + lane;
        if (EPI == EPI_RESID_F32) {  // residual rows of this CTA's first owned columns
            const int lo = (z * BN) / S;
            load_resid(p, n0 + lo, tm * BM + fl, xr0);
        }
        if (!mbar_wait(smem_u32(accf), 0u, abort_flag)) *ep_fail = 1;
        tc_fence_after();
    }

    // phase 0: every CTA of the cluster has finished its MMAs (stage rings are free)
    cluster_sync_all();
    if (warp < 4) {
        const bool ok = (*ep_fail == 0) && !*abort_flag;
        if (ok) {
            const int fl = warp * 32 + lane;
            const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
            const uint32_t red_s = smem_u32(red);
            const int ncols = min(BN, ((p.T - n0) + 31) / 32 * 32);
            for (int c0 = 0; c0 < ncols; c0 += 32) {
                uint32_t r[32];
                TMEM_LD32(trow + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int c = c0 + j;
                    const int o = ((c + 1) * S - 1) / BN;  // owner: columns [o BN / S, (o+1) BN / S)
                    const int lo = (o * BN) / S;
                    const uint32_t dst = mapa_shared(red_s + (uint32_t)(((z * WMAX + (c - lo)) * 128 + fl) * 4), (uint32_t)o);
                    st_cluster_f32(dst, __uint_as_float(r[j]));
                }
            }
        }
    }
    // phase 1: all partials have landed in their owners' shared memory
    cluster_sync_all();
    if (warp < 4) {
        const bool ok = (*ep_fail == 0) && !*abort_flag;
        if (!ok) {
            if (threadIdx.x == 0) atomicOr(p.status, QW_DEV_TIMEOUT);
        } else {
            const int fl = warp * 32 + lane;
            const int lo = (z * BN) / S, hi = ((z + 1) * BN) / S;
            for (int cc = lo; cc < hi; cc += 32) {
                const int w = min(32, hi - cc);
                const int tok0 = n0 + cc;
                if (tok0 >= p.T) break;
                const int ntok = min(w, p.T - tok0);
                if (EPI == EPI_RESID_F32) {
                    if (cc > lo) load_resid(p, tok0, tm * BM + fl, xr0);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j >= ntok) break;
                        float v = xr0[j];
                        for (int s = 0; s < S; ++s) v += red[(s * WMAX + (cc - lo) + j) * 128 + fl];
                        p.out_f32[(size_t)(tok0 + j) * p.ld_out + tm * BM + fl] = v;
                    }
                } else {
                    RopeRegs rr;
                    if (EPI == EPI_QKV_HEADS && tm < p.n_heads + p.n_kv) load_rope(p, tpos, cc, ntok, rr);
                    for (int j = 0; j < w; ++j) {
                        float v = 0.f;
                        for (int s = 0; s < S; ++s) v += red[(s * WMAX + (cc - lo) + j) * 128 + fl];
                        if (EPI == EPI_QKV_HEADS)
                            reinterpret_cast<f16*>(E)[j * EPH + fl] = __float2half_rn(v);
                        else
                            E[j * EP + fl] = v;
                    }
                    named_bar_epi();
                    if (EPI == EPI_QKV_HEADS)
                        epi_heads(p, reinterpret_cast<const f16*>(E), nws, tdst, rr, tok0, cc, ntok, tm);
                    else
                        epi_silu(p, E, tok0, ntok, tm);
                    named_bar_epi();
                }
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
}

namespace {

template <int BN, int EPI>
void fill_params(GemmKParams& p, const GemmArgs& a) {
    p = GemmKParams{};
    p.a_row0 = a.a_row0;
    p.b_row0 = a.b_row0;
    p.K = a.K;
    p.T = a.T;
    p.ld_out = a.ld_out;
    p.out_f32 = a.out_f32;
    p.out_h = a.out_h;
    p.logits = a.logits;
    p.best = a.best;
    p.status = a.status;
    p.q_out = a.q_out;
    p.q_norm = a.q_norm;
    p.k_norm = a.k_norm;
    p.eps = a.eps;
    p.rope_cos = a.rope_cos;
    p.rope_sin = a.rope_sin;
    p.tv = a.tv;
    p.kv = a.kv;
    p.layer = a.layer;
    p.n_heads = a.n_heads;
    p.n_kv = a.n_kv;
    p.dbg_pos = a.dbg_pos;
    p.dbg_slot = a.dbg_slot;
    p.tiles_m = a.M / BM;
    p.tiles_n = (a.T + BN - 1) / BN;
}

template <typename K>
cudaError_t set_smem(K kern, int bytes, bool& done) {
    if (done) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done = true;
    return e;
}

// Largest cluster size <= want for which all `clusters` clusters are co-resident (the
// device's count of simultaneously active clusters per size is probed once and cached);
// 1 when none is.
template <int BN, int EPI>
int cluster_fit(int want, int clusters, int smem, cudaStream_t st) {
    static int max_active[9] = {0};  // by cluster size; 0: not probed
    static bool probed = false;
    if (!probed) {
        probed = true;
        for (int s = 2; s <= 8; ++s) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(s);
            cfg.blockDim = dim3(GEMM_THREADS);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = st;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = s;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, k_gemm_cl<BN, EPI>, &cfg) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            max_active[s] = n;
        }
    }
    for (int s = std::min(want, 8); s >= 2; --s)
        if (max_active[s] >= clusters) return s;
    return 1;
}

template <int BN, int EPI>
cudaError_t gemm_go(const LaunchCtx& c, const GemmArgs& a, int bn_idx) {
    using CC = GemmCfg<BN, EPI, 1>;  // cluster split-K kernel
    using CT = GemmCfg<BN, EPI, 2>;  // persistent kernel
    using CP = GemmCfg<BN, EPI, 2, 2>;  // persistent kernel on CTA pairs
    static_assert(CC::SMEM <= SMEM_BUDGET && CT::SMEM <= SMEM_BUDGET && CP::SMEM <= SMEM_BUDGET,
                  "shared memory budget");
    static_assert(CC::STAGES >= 3 && CT::STAGES >= 3 && CP::STAGES >= 3, "pipeline depth");
    GemmKParams p;
    fill_params<BN, EPI>(p, a);
    const int tiles = p.tiles_m * p.tiles_n;
    const int sms = a.num_sms > 0 ? a.num_sms : 148;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (c.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (c.counter) ++*c.counter;
    if constexpr (EPI != EPI_ARGMAX) {
        int splits = 1;
        if (tiles * 2 <= sms) {
            splits = std::min(std::min(sms / tiles, 8), std::max((a.K / BK) / 4, 1));
            // the partials of all splits must fit in one CTA's stage ring
            while (splits > 1 && splits * 128 * ((BN + splits - 1) / splits) * 4 > CC::STAGES * CC::STAGE_BYTES)
                --splits;
        }
        if (splits > 1) {
            static bool done = false;
            cudaError_t e = set_smem(k_gemm_cl<BN, EPI>, CC::SMEM, done);
            if (e != cudaSuccess) return e;
            splits = cluster_fit<BN, EPI>(splits, tiles, CC::SMEM, c.stream);
        }
        if (splits > 1) {
            p.splits = splits;
            p.units = tiles;
            attr[na].id = cudaLaunchAttributeClusterDimension;
            attr[na].val.clusterDim.x = splits;
            attr[na].val.clusterDim.y = 1;
            attr[na].val.clusterDim.z = 1;
            ++na;
            cfg.gridDim = dim3(tiles * splits);
            cfg.blockDim = dim3(GEMM_THREADS);
            cfg.dynamicSmemBytes = CC::SMEM;
            cfg.attrs = attr;
            cfg.numAttrs = na;
            return cudaLaunchKernelEx(&cfg, k_gemm_cl<BN, EPI>, *a.tmA, a.tmB[bn_idx], p);
        }
    }
    p.splits = 1;
    if constexpr (QW_GEMM_PAIR && BN >= 128 && EPI != EPI_ARGMAX) {
        if (p.tiles_m % 2 == 0 && sms >= 2) {
            // 256-row tiles on CTA pairs; each CTA loads half of the token tile (map bn_idx - 1
            // has boxes of BN / 2 rows)
            static bool done_p = false;
            cudaError_t e = set_smem(k_gemm_tc<BN, EPI, true>, CP::SMEM, done_p);
            if (e != cudaSuccess) return e;
            p.units = tiles / 2;
            attr[na].id = cudaLaunchAttributeClusterDimension;
            attr[na].val.clusterDim.x = 2;
            attr[na].val.clusterDim.y = 1;
            attr[na].val.clusterDim.z = 1;
            ++na;
            cfg.gridDim = dim3(2 * std::min(p.units, sms / 2));
            cfg.blockDim = dim3(GEMM_TC_THREADS);
            cfg.dynamicSmemBytes = CP::SMEM;
            cfg.attrs = attr;
            cfg.numAttrs = na;
            return cudaLaunchKernelEx(&cfg, k_gemm_tc<BN, EPI, true>, *a.tmA, a.tmB[bn_idx - 1], p);
        }
    }
    static bool done = false;
    cudaError_t e = set_smem(k_gemm_tc<BN, EPI, false>, CT::SMEM, done);
    if (e != cudaSuccess) return e;
    p.units = tiles;
    cfg.gridDim = dim3(std::min(tiles, sms));
    cfg.blockDim = dim3(GEMM_TC_THREADS);
    cfg.dynamicSmemBytes = CT::SMEM;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, k_gemm_tc<BN, EPI, false>, *a.tmA, a.tmB[bn_idx], p);
}

template <int EPI>
cudaError_t gemm_bn(const LaunchCtx& c, const GemmArgs& a) {
    if (a.T <= 64) return gemm_go<64, EPI>(c, a, 0);
    if (a.T <= 128) return gemm_go<128, EPI>(c, a, 1);
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
        case EPI_QKV_HEADS: return gemm_bn<EPI_QKV_HEADS>(c, a);
        case EPI_RESID_F32: return gemm_bn<EPI_RESID_F32>(c, a);
        case EPI_SILU_MUL: return gemm_bn<EPI_SILU_MUL>(c, a);
        case EPI_ARGMAX: return gemm_bn<EPI_ARGMAX>(c, a);
        default: return cudaErrorInvalidValue;
    }
}
