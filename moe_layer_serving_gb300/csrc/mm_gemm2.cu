// mm_gemm2.cu -- the large-input grouped GEMM on CTA pairs (2-SM MMA).
//
// What bounds the one-CTA grouped GEMM is the bytes each SM's TMA writes into
// shared memory per stage: 16 KB of token rows and 32 KB of weights (the FP4
// weights take a byte per element once unpacked for the MMA), against 512
// cycles of MMA work.  Here the two CTAs of a cluster run one MMA over both
// SMs (tcgen05 cta_group::2): M = 256 token rows, 128 from each CTA's shared
// memory, and N = 256 weight rows, likewise 128 from each.  Each SM then takes
// in 32 KB a stage for the same 512 cycles of tensor work, and six stages fit
// where four did.
//
// A unit is (pair of token tiles of one expert, weight block pair): GEMM1
// units put the gate rows of 128 I-columns in CTA 0 and the up rows in CTA 1,
// GEMM2 units the two 128-row halves of 256 output features.  Each CTA holds
// its tile's 128 rows of the accumulator over all 256 columns, so its
// epilogue is the one-CTA kernel's (SwiGLU pairs gate column c with up column
// 128 + c in one thread).  An expert with an odd number of tiles leaves the
// second CTA without a tile in its last pair: that CTA loads only its half of
// the weights, and its accumulator rows are never read.  Such pairs cost a
// whole tile of MMA work each, so by default the large path launches this
// kernel after the one-CTA kernel and the tile scan picks the one that runs
// (GemmArgs::select, num_tiles[3]).
//
// Roles: warp 0 lane 0 = token-side producer (own token tile and its
// scales), warp 10 lane 0 = weight-side producer (own weight half and both
// halves' weight scales -- the MMA reads the weight scales of all 256 columns
// in each CTA's tensor memory), in both CTAs, every copy completing on CTA 0's
// barrier; warp 1 = tensor-memory owner and, in CTA 0, the MMA issuer (in CTA
// 1 it only takes the unit numbers out of the ring); warps 2..9 = epilogue,
// which in CTA 1 releases each drained accumulator with one relaxed remote
// arrive per warp on CTA 0's peer_tmem_empty (relaying through a warp of CTA 1,
// or arriving from every thread with release semantics, held the pair's MMAs
// ~1,700 / ~2,000 cycles a unit).  Unit numbers are drawn by CTA 0's
// token-side producer and handed to CTA 1's, so both run the same sequence.
// Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mm_gemm.cuh"

namespace mm {
namespace {

constexpr int kStages2 = 6;
constexpr int kA2Bytes = kTokTile * kKStep;                       // 128 token rows x 128 K
constexpr int kSF2Off = kA2Bytes + kWBoxBytes;                    // scales after this CTA's weight rows
constexpr int kStage2Bytes = (kSF2Off + 3 * kSFBytes + 1023) / 1024 * 1024;
constexpr int kStageRegion2 = kStages2 * kStage2Bytes;
constexpr int kSmem2Bytes = kStageRegion2 + kBarBlock + 1024;
static_assert(kStages2 <= kMaxStages, "barrier block holds eight stages");
static_assert(kSmem2Bytes <= 232448, "shared memory per block");
static_assert(kColSF + kStages2 * kSFSlotCols <= kTmemCols, "scale slots fit the allocation");


// Number u -> unit; this CTA's tile is the pair's first (rank 0) or second
// (rank 1, -1 when the expert's tile count was odd).
__device__ __forceinline__ bool decode2(const GemmArgs& g, int npairs, int u, uint32_t rank, Unit& un)
{
    const int nb1 = g.I / kTile, nb2 = g.H / (2 * kTile);
    const int units1 = npairs * nb1, units2 = npairs * nb2;
    if (u < 0 || u >= units1 + units2) return false;
    int st;
    if (u < units1) {
        un.phase = 1;
        st = u / nb1;
        un.blk = u % nb1;
    } else {
        un.phase = 2;
        st = (u - units1) / nb2;
        un.blk = (u - units1) % nb2;
    }
    const int t0 = g.st_tile[2 * st];
    const int t = g.st_tile[2 * st + rank];
    un.expert = g.tile_expert[t0];
    un.tile = t;
    un.row0 = t >= 0 ? g.tile_row0[t] : 0;
    un.rows = t >= 0 ? g.tile_rows[t] : 0;
    if (!MM_CHECK(un.expert >= 0 && un.expert < g.P && un.row0 >= 0 && un.rows >= 0 && un.rows <= 128 &&
                      un.row0 + un.rows <= g.rows_cap,
                  g.status, kSiteGemmTile))
        return false;
    un.tbox = un.rows <= 16 ? 0 : (un.rows <= 32 ? 1 : (un.rows <= 64 ? 2 : 3));
    un.nw = 2;
    if (un.phase == 1) {
        un.ksteps = g.H / kKStep;
        un.wz = (un.expert * nb1 + un.blk) * un.ksteps * 2;
        un.m0 = 0;
    } else {
        un.m0 = 2 * un.blk * kTile;
        un.ksteps = g.I / kKStep;
        un.wz = (un.expert * nb2 + un.blk) * un.ksteps * 2;
    }
    return true;
}

// kSide: kSideTokens (draws or receives the unit numbers, waits for GEMM1
// results before a GEMM2 unit) or kSideWeights (takes the numbers out of the
// CTA's ring).  In CTA 0 each side arrives on the stage's full barrier with
// the bytes of its side in both CTAs.
template <int kSide>
__device__ __forceinline__ void producer2(const GemmMaps& maps, const GemmArgs& g, int npairs, const GemmSmem& s,
                                          uint32_t rank)
{
    constexpr bool kTok = kSide == kSideTokens;
    const uint64_t pol_w = g.keep_weights ? policy_evict_normal() : policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    int armed[kStages2];
    for (int i = 0; i < kStages2; ++i) armed[i] = -1;
    Unit un;
    UnitQueue q, box;
    for (;;) {
        int u;
        const bool got = kTok ? push_unit(g, s, q, u, &box, rank) : pop_unit(g, s, q, u);
        if (!got || *s.abort_flag || !decode2(g, npairs, u, rank, un)) break;
        const bool has = un.rows > 0;
        const CUtensorMap* wmap = un.phase == 1 ? &maps.w1_one : &maps.w2_one;
        const CUtensorMap* amap = un.phase == 1 ? &maps.xq[un.tbox] : &maps.hq[un.tbox];
        if (kTok && un.phase == 2 && has) {
            const int need = g.I / kTile + (g.fault == kFaultGemmDependency ? 1 : 0);
            if (ld_acquire(&g.done1[un.tile]) < need) {
                const uint64_t t0 = globaltimer();
                while (ld_acquire(&g.done1[un.tile]) < need) {
                    if (*s.abort_flag) break;
                    if (globaltimer() - t0 > kWaitLimitNs) {
                        latch_error(g.status, MM_ERR_TIMEOUT, kSiteProducerDone1);
                        *s.abort_flag = 1;
                        break;
                    }
                }
            }
            fence_proxy_async_global();
            if (*s.abort_flag) break;
        }
        // Every copy of a stage, in either CTA, completes on CTA 0's full
        // barrier (tile loads whose mbarrier may be the pair's other CTA's), so
        // CTA 0's barrier counts the bytes of both: CTA 0's MMA waits on it
        // alone.  (CTA 1 reporting its own landed stages by remote arrives
        // measured 1.8x slower: the MMA warp woke late on each of them.)
        uint32_t bytes = 2 * (kWBoxTxBytes + 2 * kSFBytes);
        if (kTok) {
            bytes = has ? (kBBox << un.tbox) * kKStep + kSFBytes : 0;
            if (rank == 0) {
                Unit peer;
                if (!decode2(g, npairs, u, 1, peer)) break;
                bytes += peer.rows > 0 ? (kBBox << peer.tbox) * kKStep + kSFBytes : 0;
            }
        }
        const CUtensorMap* asf_map = un.phase == 1 ? &maps.xs_sf : &maps.hs_sf;
        const CUtensorMap* wsf_map = un.phase == 1 ? &maps.w1_sf : &maps.w2_sf;
        // this CTA's member of each stage's block pair
        const uint8_t* wblk = (un.phase == 1 ? g.w1 : g.w2) + static_cast<int64_t>(un.wz + rank) * kWBoxTxBytes;
        if (!kTok && kPrefetch > 0) {
            for (int j = 1; j < kPrefetch && j < un.ksteps; ++j)
                prefetch_l2(wblk + static_cast<int64_t>(2 * j) * kWBoxTxBytes, kWBoxTxBytes);
        }
        for (int ks = 0; ks < un.ksteps; ++ks) {
            if (!kTok && kPrefetch > 0 && ks + kPrefetch < un.ksteps)
                prefetch_l2(wblk + static_cast<int64_t>(2 * (ks + kPrefetch)) * kWBoxTxBytes, kWBoxTxBytes);
            if (!mbar_wait(&s.empty[stage], phase ^ 1u, g.status, s.abort_flag, kSiteProducerEmpty)) break;
            uint8_t* st = s.stages + stage * kStage2Bytes;
            uint8_t* sf = st + kSF2Off;
            const int wz = un.wz + 2 * ks;
            const uint32_t bar = peer_addr(&s.full[stage], 0);
            if (rank == 0) {
                mbar_arrive_expect_tx(&s.full[stage], bytes);
                armed[stage] = static_cast<int>(phase);
            }
            if (kTok) {
                if (has) {
                    tma_load_2d_pair(st, amap, ks * kKStep, un.row0, bar, pol_a);
                    tma_load_2d_pair(sf, asf_map, 0, 2 * (un.tile * un.ksteps + ks), bar, pol_a);
                }
            } else {
                tma_load_3d_pair(st + kA2Bytes, wmap, 0, 0, wz + static_cast<int>(rank), bar, pol_w);
                tma_load_2d_pair(sf + kSFBytes, wsf_map, 0, 2 * wz, bar, pol_w);
            }
            if (++stage == kStages2) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (*s.abort_flag) {
        // (one deadline for all stages: a stage the other side never armed
        // does not complete although this side's copies landed)
        const uint64_t t0 = globaltimer();
        for (int i = 0; i < kStages2; ++i) {
            if (armed[i] < 0) continue;
            while (!mbar_try_wait(&s.full[i], static_cast<uint32_t>(armed[i])))
                if (globaltimer() - t0 > kWaitLimitNs / 4) break;
        }
    }
}

// Warp 1 of CTA 0: the pair's MMAs.  A stage is used once both CTAs' copies
// landed (all of them complete on CTA 0's full barrier); its scales go to
// tensor memory by 2-SM copies (each CTA's own shared memory into its own
// tensor memory), then four MMAs of K = 32, and a commit frees the stage in
// both CTAs.
__device__ __forceinline__ void mma2_loop(const GemmArgs& g, int npairs, const GemmSmem& s, uint32_t tmem)
{
    const uint64_t a_desc0 = desc_kmajor_sw128(s.stages);
    const uint64_t b_desc0 = desc_kmajor_sw128(s.stages + kA2Bytes);
    const uint64_t sf_desc0 = desc_sf(s.stages + kSF2Off);
    static_assert(kStages2 * kStage2Bytes + 1024 < (1 << 18), "descriptor address field");
    constexpr uint64_t kStageDesc = kStage2Bytes >> 4, kSfDesc = kSFBytes >> 4;
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool aborted = false;
    Unit un;
    UnitQueue q;
    const int lane = threadIdx.x & 31;
    for (;;) {
        const bool got = mbar_wait(&s.ufull[q.slot], q.phase, g.status, s.abort_flag, kSiteUnitQueue);
        if (!__all_sync(0xFFFFFFFFu, got)) break;
        const int u = s.uring[q.slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.uempty[q.slot]);
        q.advance();
        if (*s.abort_flag || !decode2(g, npairs, u, 0, un)) break;
        // both CTAs' accumulators drained by their epilogues
        const bool drained =
            mbar_wait(s.tmem_empty, acc_phase ^ 1u, g.status, s.abort_flag, kSiteMmaTmemEmpty) &&
            mbar_wait_cluster(s.peer_tmem_empty, acc_phase ^ 1u, g.status, s.abort_flag, kSiteMmaTmemEmpty);
        if (!__all_sync(0xFFFFFFFFu, drained)) {
            aborted = true;
            break;
        }
        tc_fence_after();
        const uint32_t id0 = idesc_e4m3_e2m1(256, 0, 256), id1 = idesc_e4m3_e2m1(256, 1, 256);
        const uint32_t id2 = idesc_e4m3_e2m1(256, 2, 256), id3 = idesc_e4m3_e2m1(256, 3, 256);
        for (int ks = 0; ks < un.ksteps; ++ks) {
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&s.full[stage], phase, g.status, s.abort_flag, kSiteMmaFull))) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint64_t off = static_cast<uint64_t>(stage) * kStageDesc;
            const uint64_t ad = a_desc0 + off, bd = b_desc0 + off, sd = sf_desc0 + off;
            const uint32_t t_sfa = tmem + kColSF + stage * kSFSlotCols, t_sfb = t_sfa + kColSFB;
            if (elect_one()) {
                tc_cp2_32x128b_x4(t_sfa, sd);
                tc_cp2_32x128b_x4(t_sfb, sd + kSfDesc);
                tc_cp2_32x128b_x4(t_sfb + 4, sd + 2 * kSfDesc);
                if (ks == 0)
                    mma2_mxf8f6f4<false>(tmem, ad, bd, id0, t_sfa, t_sfb);
                else
                    mma2_mxf8f6f4<true>(tmem, ad, bd, id0, t_sfa, t_sfb);
                mma2_mxf8f6f4<true>(tmem, ad + 2, bd + 2, id1, t_sfa, t_sfb);
                mma2_mxf8f6f4<true>(tmem, ad + 4, bd + 4, id2, t_sfa, t_sfb);
                mma2_mxf8f6f4<true>(tmem, ad + 6, bd + 6, id3, t_sfa, t_sfb);
                tc_commit2_mc(&s.empty[stage], 0x3);
            }
            __syncwarp();
            if (++stage == kStages2) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (aborted || *s.abort_flag) break;
        if (elect_one()) tc_commit2_mc(s.tmem_full, 0x3);
        __syncwarp();
        acc_phase ^= 1u;
    }
    if (*s.abort_flag) {
        if (elect_one()) {
            tc_commit2_mc(s.drain, 0x1);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(s.drain, 0))
                if (globaltimer() - t0 > kWaitLimitNs / 4) break;
        }
        __syncwarp();
    }
}

// Warp 1 of CTA 1: takes the unit numbers out of the ring (one of its
// consumers), nothing else.
__device__ __forceinline__ void unit_sink_loop(const GemmArgs& g, int npairs, const GemmSmem& s)
{
    const int lane = threadIdx.x & 31;
    Unit un;
    UnitQueue q;
    for (;;) {
        const bool got = mbar_wait(&s.ufull[q.slot], q.phase, g.status, s.abort_flag, kSiteUnitQueue);
        if (!__all_sync(0xFFFFFFFFu, got)) break;
        const int u = s.uring[q.slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.uempty[q.slot]);
        q.advance();
        if (*s.abort_flag || !decode2(g, npairs, u, 1, un)) break;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm2_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs g)
{
    // the batch went to the one-CTA kernel (launched before this one): every
    // CTA of every pair reads the same choice and returns before any barrier
    if (g.select == 2 && g.num_tiles[3] == 0) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const GemmSmem s = gemm_smem(smem, smem + kStageRegion2);
    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages2; ++i) {
            mbar_init(&s.full[i], 2);          // CTA 0's: both producer sides arrive
            mbar_init(&s.empty[i], 1);
        }
        mbar_init(s.tmem_full, 1);
        mbar_init(s.tmem_empty, kEpiThreads);
        mbar_init(s.peer_tmem_empty, kEpiThreads / 32);   // one arrive per epilogue warp of CTA 1
        mbar_init(s.drain, 1);
        for (int i = 0; i < kURing; ++i) {
            mbar_init(&s.ufull[i], 1);
            mbar_init(&s.uempty[i], 2 + kEpiThreads);
            mbar_init(&s.inbox_full[i], 1);
            mbar_init(&s.inbox_free[i], 1);
        }
        *s.abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&maps.w1_one);
        prefetch_tmap(&maps.w2_one);
    }
    if (warp == 1) {
        tmem_alloc2(s.tmem_slot, kTmemCols);      // collectively: the same columns in both CTAs
        tmem_relinquish2();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *s.tmem_slot;
    const int npairs = g.num_tiles[2];
    if (warp == 0) {
        if (lane == 0) producer2<kSideTokens>(maps, g, npairs, s, rank);
    } else if (warp == kWProdWarp) {
        if (lane == 0) producer2<kSideWeights>(maps, g, npairs, s, rank);
    } else if (warp == 1) {
        if (rank == 0)
            mma2_loop(g, npairs, s, tmem);
        else
            unit_sink_loop(g, npairs, s);
    } else {
        epilogue_loop(g, s, tmem, [&](int u, Unit& un) { return decode2(g, npairs, u, rank, un); },
                      rank == 1 ? peer_addr(s.peer_tmem_empty, 0) : 0u);
    }
    // neither CTA frees tensor memory or exits before the pair is done with it
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem, kTmemCols);
    }
}

// clusters of two the GPU holds at once with one CTA per SM (-1 = none)
int g_clusters2[64];

}  // namespace

cudaError_t gemm2_prepare(int dev)
{
    cudaError_t e = cudaFuncSetAttribute(gemm2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem2Bytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && g_clusters2[dev] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem2Bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm2_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        g_clusters2[dev] = n > 0 ? n : -1;
    }
    return cudaSuccess;
}

bool gemm2_usable(const mm_ctx* c)
{
    // every GEMM2 unit a full pair of 128-row weight blocks
    return c->gemm_2sm != 0 && c->dev >= 0 && c->dev < 64 && g_clusters2[c->dev] > 0 && c->H % (2 * kTile) == 0;
}

cudaError_t launch_gemm2(const mm_ctx* c, cudaStream_t s, int select)
{
    GemmArgs g;
    fill_gemm_args(c, &g);
    g.select = select;
    // an expert's pairs re-read its weight blocks: the normal L2 policy (with
    // evict-first a 16-expert prefill read 2.1 GB from DRAM instead of 0.8)
    g.keep_weights = 1;
    const int clusters = g_clusters2[c->dev] < c->sms / 2 ? g_clusters2[c->dev] : c->sms / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem2Bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm2_kernel, c->maps, g);
}

}  // namespace mm
