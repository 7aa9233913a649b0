// mm_gemm.cuh -- the persistent grouped block-scaled GEMM machinery of the
// fused MoE forward on sm_103a, shared by the large-input kernel and the fused
// small-input kernel.
//
// Both GEMMs run "weights as A": the MMA's M = 128 weight rows (e2m1, the
// packed MXFP4 operand, unpacked to one byte per element in shared memory by
// the TMA), N = up to 112 dispatched token rows of one physical expert (e4m3),
// K in stages of 128, one e8m0 scale per 32 along K for both operands
// (tcgen05.mma kind::mxf8f6f4 block_scale, fp32 accumulators in tensor memory).
//
//   GEMM1 unit (tile, n-block): gate rows [nb*128, +128) and up rows
//       [I + nb*128, +128) of W1[p] against the tile's activation rows; the
//       epilogue forms h = silu(gate) * up and quantises h to MXFP8 along I
//       (one 32-column block per warp), writing hq/hs for the tile.
//   GEMM2 unit (tile, m-pair): W2[p] rows [2m*128, +256) against hq of the
//       tile; the epilogue writes y rows in bf16.
//
// A persistent CTA walks units u = first, first + stride, ...; all GEMM1 units
// precede all GEMM2 units, and a GEMM2 unit waits (bounded) until the GEMM1
// units of its tile have published hq.  Warp roles: 0 = TMA producer, 1 =
// tensor-memory owner + MMA issuer, 2..5 = epilogue.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {

constexpr int kThreads = 192;
constexpr int kEpiWarp0 = 2;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: two accumulator buffers of 2 x kTileN fp32 columns (one per A
// tile), then the scale factors of the current stage.
constexpr uint32_t kAccCols = 2 * kTileN;
constexpr uint32_t kColSFA0 = 2 * kAccCols, kColSFA1 = kColSFA0 + 4, kColSFB = kColSFA0 + 8;
static_assert(kColSFB + 4 <= kTmemCols, "accumulators and scale factors must fit in TMEM");

struct Unit {
    int phase;      // 1 or 2
    int tile;
    int blk;        // n-block (GEMM1) or m-pair (GEMM2)
    int expert;
    int row0;       // first dispatch row of the tile
    int rows;       // valid rows in the tile
    int n;          // MMA N: rows rounded up to 16
    int na;         // A tiles (1 or 2)
    int ksteps;
    int arow[2];    // first weight row of each A tile (global row of the stacked weights)
    int sfrb[2];    // scale-tile row block of each A tile
};

// Token tiles the GEMMs run over (generic pointers: global or shared memory).
struct TileView {
    const int* expert;
    const int* row0;
    const int* rows;
    int ntiles;
};

__device__ __forceinline__ bool decode_unit(const GemmArgs& g, const TileView& tv, int u, Unit& un)
{
    const int ntiles = tv.ntiles;
    const int nb1 = g.I / kTile;
    const int nb2 = (g.H + 2 * kTile - 1) / (2 * kTile);
    const int units1 = (g.phases & 1) ? ntiles * nb1 : 0;
    const int units2 = (g.phases & 2) ? ntiles * nb2 : 0;
    if (u >= units1 + units2) return false;
    if (u < units1) {
        un.phase = 1;
        un.tile = u / nb1;
        un.blk = u % nb1;
    } else {
        un.phase = 2;
        un.tile = (u - units1) / nb2;
        un.blk = (u - units1) % nb2;
    }
    un.expert = tv.expert[un.tile];
    un.row0 = tv.row0[un.tile];
    un.rows = tv.rows[un.tile];
    un.n = (un.rows + 15) & ~15;
    if (un.phase == 1) {
        un.na = 2;
        un.ksteps = g.H / kKStep;
        const int base = un.expert * 2 * g.I;
        un.arow[0] = base + un.blk * kTile;
        un.arow[1] = base + g.I + un.blk * kTile;
    } else {
        const int r0 = 2 * un.blk * kTile;
        un.na = (r0 + kTile < g.H) ? 2 : 1;
        un.ksteps = g.I / kKStep;
        un.arow[0] = un.expert * g.H + r0;
        un.arow[1] = un.expert * g.H + r0 + kTile;
    }
    un.sfrb[0] = un.arow[0] / kTile;
    un.sfrb[1] = un.arow[1] / kTile;
    return true;
}

__device__ __forceinline__ int ld_acquire(const int* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// shared-memory carve-up of the GEMM machinery (base aligned to 1024 bytes)
struct GemmSmem {
    uint8_t* stages;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tmem_full;
    uint64_t* tmem_empty;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
};
constexpr int kGemmSmemBytes = kStages * kStageBytes + 256;   // stages + barriers

__device__ __forceinline__ GemmSmem gemm_smem(uint8_t* smem)
{
    GemmSmem s;
    s.stages = smem;
    s.full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    s.empty = s.full + kStages;
    s.tmem_full = s.empty + kStages;      // [2], one per accumulator buffer
    s.tmem_empty = s.tmem_full + 2;       // [2]
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.tmem_empty + 2);
    s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
    return s;
}

// All threads: barriers, tensor-memory allocation (warp 1); returns the TMEM base.
__device__ __forceinline__ uint32_t gemm_setup(const GemmSmem& s, const GemmMaps& maps)
{
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s.tmem_full[b], 1);
            mbar_init(&s.tmem_empty[b], 128);
        }
        *s.abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&maps.w1);
        prefetch_tmap(&maps.w2);
        prefetch_tmap(&maps.xq);
        prefetch_tmap(&maps.hq);
    }
    if (warp == 1) {
        tmem_alloc(s.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return *s.tmem_slot;
}

// All threads: wait for every role, free tensor memory.
__device__ __forceinline__ void gemm_teardown(uint32_t tmem)
{
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// All threads: each warp runs its role over units first_unit, +unit_stride, ...
__device__ __forceinline__ void gemm_roles(const GemmMaps& maps, const GemmArgs& g, const TileView& tv,
                                           const GemmSmem& s, uint32_t tmem, int first_unit, int unit_stride)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* smem = s.stages;
    uint64_t* full = s.full;
    uint64_t* empty = s.empty;
    uint64_t* tmem_full = s.tmem_full;
    uint64_t* tmem_empty = s.tmem_empty;
    volatile int* abort_flag = s.abort_flag;
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            int armed[kStages];
            for (int s = 0; s < kStages; ++s) armed[s] = -1;
            Unit un;
            for (int u = first_unit; decode_unit(g, tv, u, un) && !*abort_flag; u += unit_stride) {
                const CUtensorMap* wmap = un.phase == 1 ? &maps.w1 : &maps.w2;
                const CUtensorMap* amap = un.phase == 1 ? &maps.xq : &maps.hq;
                const uint8_t* wsf = un.phase == 1 ? g.w1_sf : g.w2_sf;
                const uint8_t* asf = un.phase == 1 ? g.xs_t : g.hs_t;
                if (un.phase == 2) {
                    const int need = g.I / kTile;
                    if (ld_acquire(&g.done1[un.tile]) < need) {
                        const uint64_t t0 = globaltimer();
                        while (ld_acquire(&g.done1[un.tile]) < need) {
                            if (*abort_flag) break;
                            if (globaltimer() - t0 > kWaitLimitNs) {
                                latch_error(g.status, MM_ERR_TIMEOUT, kSiteProducerDone1);
                                *abort_flag = 1;
                                break;
                            }
                        }
                    }
                    fence_proxy_async_global();
                    if (*abort_flag) break;
                }
                const int nbox = un.n / kBBox;
                const uint32_t bytes = un.na * kATileTxBytes + nbox * kBBox * kKStep + (un.na + 1) * kSFBytes;
                for (int ks = 0; ks < un.ksteps; ++ks) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, g.status, abort_flag, kSiteProducerEmpty)) break;
                    uint8_t* st = smem + stage * kStageBytes;
                    uint8_t* sf = st + 2 * kATileBytes + kBTileBytes;
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    armed[stage] = static_cast<int>(phase);
                    for (int a = 0; a < un.na; ++a) {
                        tma_load_3d(st + a * kATileBytes, wmap, 0, 0, un.sfrb[a] * un.ksteps + ks, &full[stage],
                                    pol_w);
                        bulk_load(sf + a * kSFBytes, wsf + (static_cast<int64_t>(un.sfrb[a]) * un.ksteps + ks) * kSFBytes,
                                  kSFBytes, &full[stage]);
                    }
                    for (int bx = 0; bx < nbox; ++bx)
                        tma_load_2d(st + 2 * kATileBytes + bx * kBBox * kKStep, amap, ks * kKStep,
                                    un.row0 + bx * kBBox, &full[stage], pol_a);
                    bulk_load(sf + 2 * kSFBytes,
                              asf + (static_cast<int64_t>(un.tile) * un.ksteps + ks) * kSFBytes, kSFBytes,
                              &full[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA exits
                for (int s = 0; s < kStages; ++s) {
                    if (armed[s] < 0) continue;
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(&full[s], static_cast<uint32_t>(armed[s])))
                        if (globaltimer() - t0 > kWaitLimitNs / 4) break;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_iter = 0;
            Unit un;
            for (int u = first_unit; decode_unit(g, tv, u, un) && !*abort_flag; u += unit_stride) {
                const uint32_t buf = acc_iter & 1u, acc_phase = (acc_iter >> 1) & 1u;
                if (!mbar_wait(&tmem_empty[buf], acc_phase ^ 1u, g.status, abort_flag, kSiteMmaTmemEmpty)) break;
                tc_fence_after();
                for (int ks = 0; ks < un.ksteps; ++ks) {
                    if (!mbar_wait(&full[stage], phase, g.status, abort_flag, kSiteMmaFull)) break;
                    tc_fence_after();
                    uint8_t* st = smem + stage * kStageBytes;
                    uint8_t* sf = st + 2 * kATileBytes + kBTileBytes;
                    tc_cp_32x128b_x4(tmem + kColSFA0, desc_sf(sf));
                    if (un.na == 2) tc_cp_32x128b_x4(tmem + kColSFA1, desc_sf(sf + kSFBytes));
                    tc_cp_32x128b_x4(tmem + kColSFB, desc_sf(sf + 2 * kSFBytes));
                    const uint64_t bdesc = desc_kmajor_sw128(st + 2 * kATileBytes);
#pragma unroll
                    for (int kk = 0; kk < kKStep / 32; ++kk) {
                        const uint32_t idesc = idesc_e2m1_e4m3(static_cast<uint32_t>(un.n), kk);
                        for (int a = 0; a < un.na; ++a) {
                            const uint64_t adesc = desc_kmajor_sw128(st + a * kATileBytes);
                            mma_mxf8f6f4(tmem + buf * kAccCols + a * kTileN, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                                         tmem + (a == 0 ? kColSFA0 : kColSFA1), tmem + kColSFB,
                                         (ks | kk) != 0 ? 1u : 0u);
                        }
                    }
                    tc_commit(&empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (*abort_flag) break;
                tc_commit(&tmem_full[buf]);
                ++acc_iter;
            }
            if (*abort_flag) {
                // drain issued tensor-core work before the allocation is freed
                const uint32_t buf = acc_iter & 1u, acc_phase = (acc_iter >> 1) & 1u;
                tc_commit(&tmem_full[buf]);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&tmem_full[buf], acc_phase))
                    if (globaltimer() - t0 > kWaitLimitNs / 4) break;
            }
        }
    } else {
        // --------------------------------------------------------------- epilogue
        const int q = warp & 3;                  // tensor-memory lane quarter of this warp
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        uint32_t acc_iter = 0;
        Unit un;
        for (int u = first_unit; decode_unit(g, tv, u, un) && !*abort_flag; u += unit_stride) {
            const uint32_t buf = acc_iter & 1u, acc_phase = (acc_iter >> 1) & 1u;
            const uint32_t acc = tmem + lane_base + buf * kAccCols;
            if (!mbar_wait(&tmem_full[buf], acc_phase, g.status, abort_flag, kSiteEpiTmemFull)) break;
            tc_fence_after();
            if (un.phase == 1) {
                const int col = un.blk * kTile + 32 * q + lane;   // column of h (I axis)
                const int kchunks = g.I / kKStep;
                for (int c0 = 0; c0 < un.n; c0 += 16) {
                    uint32_t gr[16], ur[16];
                    tmem_ld_32x32b_x16(acc + c0, gr);
                    tmem_ld_32x32b_x16(acc + kTileN + c0, ur);
                    tmem_ld_wait();
                    // SwiGLU for 16 token columns, then their 16 warp-wide amax
                    // reductions interleaved, then codes; columns past the tile's
                    // rows are computed but not stored
                    float h[16], am[16];
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) {
                        const float gv = __uint_as_float(gr[cc]);
                        h[cc] = gv / (1.0f + __expf(-gv)) * __uint_as_float(ur[cc]);
                        am[cc] = fabsf(h[cc]);
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc)
                            am[cc] = fmaxf(am[cc], __shfl_xor_sync(0xFFFFFFFFu, am[cc], off));
                    }
                    const int cmax = min(16, un.rows - c0);
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) {
                        if (cc < cmax) {
                            const int X = mx_e4m3_exponent(am[cc]);
                            const uint32_t code = am[cc] > 0.0f ? e4m3_code(h[cc], exp2i(-X)) : 0u;
                            const int64_t row = un.row0 + c0 + cc;
                            g.hq[row * g.I + col] = static_cast<uint8_t>(code);
                            if (lane == 0)
                                g.hs_t[act_sf_offset(un.tile, c0 + cc, col / 32, kchunks)] =
                                    static_cast<uint8_t>(X + 127);
                        }
                    }
                }
            } else {
                for (int a = 0; a < un.na; ++a) {
                    const int m = (un.arow[a] - un.expert * g.H) + 32 * q + lane;   // output feature
                    for (int c0 = 0; c0 < un.n; c0 += 16) {
                        uint32_t vr[16];
                        tmem_ld_32x32b_x16(acc + a * kTileN + c0, vr);
                        tmem_ld_wait();
                        const int cmax = min(16, un.rows - c0);
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc)
                            if (cc < cmax)
                                g.y[static_cast<int64_t>(un.row0 + c0 + cc) * g.H + m] =
                                    __float2bfloat16_rn(__uint_as_float(vr[cc]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tmem_empty[buf]);
            if (un.phase == 1) {
                fence_proxy_async_global();
                __threadfence();
                epi_bar_sync();
                if (threadIdx.x == kEpiWarp0 * 32) atomicAdd(&g.done1[un.tile], 1);
            }
            ++acc_iter;
        }
    }

}

}  // namespace mm
