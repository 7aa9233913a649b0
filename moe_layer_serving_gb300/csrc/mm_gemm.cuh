// mm_gemm.cuh -- the persistent grouped block-scaled GEMM machinery of the
// fused MoE forward on sm_103a, shared by the large-input kernel and the fused
// small-input kernel.
//
// One MMA computes D[128 token rows][256 weight rows] += A . B^T over K = 32:
// A = a token tile (e4m3, K-major, one e8m0 scale per 32), B = 256 rows of
// MXFP4 weights (e2m1 unpacked to one byte per element in shared memory by the
// TMA, K-major, one e8m0 scale per 32); tcgen05.mma kind::mxf8f6f4
// block_scale, fp32 accumulators in tensor memory.  An MMA costs at least ~45
// cycles whatever its N and reaches the full rate only at N = 256 (128 cycles
// for 128 x 256 x 32), so N is always the full 256 (or 128 for a ragged last
// block of GEMM2):
//
//   GEMM1 unit (tile, n-block nb): B = gate rows [nb*128, +128) and up rows
//       [I + nb*128, +128) of W1[p]; accumulator column c holds gate and
//       column 128 + c the up projection of I-column nb*128 + c, so one thread
//       (one token row) forms h = silu(gate) * up and quantises h to MXFP8 in
//       its own registers (32-column blocks along I), writing hq/hs.
//   GEMM2 unit (tile, m-block mb): B = W2[p] rows [mb*256, +256); the
//       epilogue writes y rows in bf16.
//
// Units are handed out at run time: the producer thread of a CTA takes the
// next unit number from a global counter and passes it to the CTA's MMA and
// epilogue warps through a small ring in shared memory, so CTAs that drew
// cheaper units take more of them (GEMM1 units stream 3.5x the weight bytes of
// GEMM2 units, so a fixed round-robin split leaves some SMs a whole GEMM1 unit
// behind).  All GEMM1 units precede all GEMM2 units, and a GEMM2 unit waits
// (bounded) until the GEMM1 units of its tile have published hq.  Warp roles:
// 0 = token-side TMA producer (one lane; it also draws the units), 10 =
// weight-side TMA producer (one lane), 1 = tensor-memory owner + MMA issuer
// (the whole warp, one elected lane issuing), 2..9 = epilogue.
//
// Issuing a stage's copies takes one thread about 500 cycles (each bulk copy
// ~130, each tensor copy ~60, the expect-tx arrive and the L2 prefetch more),
// about as long as the stage's MMAs (555 cycles), so a single producer thread
// cannot get ahead of the tensor cores again after a late stage.  The producer
// is therefore split: the token side issues the token rows and their scales,
// the weight side the weight blocks, their scales and the L2 prefetch, and
// each arrives on the stage's full barrier with its own byte count.  The eight
// epilogue warps
// first drain the accumulator into registers (each warp: its 32 token rows,
// half of the columns) and release tensor memory, so the next unit's MMAs run
// while they compute.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {

constexpr int kThreads = 352;              // 11 warps
constexpr int kWProdWarp = 10;             // the weight-side producer
constexpr int kEpiWarp0 = 2;
constexpr int kEpiThreads = 256;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: accumulator [0, 256), then one scale-factor slot of 16 columns
// per pipeline stage (SFA: 4 columns, SFB: 4 columns per 128 weight rows).  A
// stage's copy into its own slot never waits for the MMAs of the stage before
// it to have read their scales.
constexpr uint32_t kColSF = 256, kSFSlotCols = 16, kColSFB = 4;

// Shared-memory pipeline geometry: token rows held per stage (the tile size
// of the kernel's token tiles) and the number of stages.  The MMA reads 128
// token rows whatever the tile size; rows past a short tile's region lie in
// the same stage's weight region and only feed accumulator rows the epilogue
// ignores.  The fused small-input kernel uses short tiles so that one more
// stage fits: with few tokens per expert its time is the weight stream's,
// set by how many bytes each SM keeps in flight.
constexpr int kBarBlock = 512;           // bytes of mbarriers and scalars after the stages

template <int kRows_, int kStages_>
struct Geom {
    static constexpr int kRows = kRows_;
    static constexpr int kStages = kStages_;
    static constexpr int kABytes = kRows * kKStep;
    static constexpr int kStageBytes = kABytes + 2 * kWBoxBytes + 4 * kSFBytes;
    static constexpr int kStageRegion = kStages * kStageBytes;
    static constexpr int kSmemBytes = kStageRegion + kBarBlock;   // stages + barriers
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static_assert(kRows % 16 == 0 && kRows <= 128, "token rows per stage");
    static_assert(kStages <= 8, "barrier block holds eight stages");
};
using GeomLarge = Geom<kTokTile, MM_STAGES>;
using GeomSmall = Geom<kSmallTile, MM_SMALL_STAGES>;

struct Unit {
    int phase;      // 1 or 2
    int tile;
    int blk;        // n-block (GEMM1) or m-block (GEMM2)
    int expert;
    int row0;       // first dispatch row of the tile
    int rows;       // valid rows in the tile
    int nw;         // weight boxes of 128 rows (1 or 2): the MMA's N = 128 * nw
    int ksteps;
    int tbox;       // token box map: 16 << tbox rows (the smallest that covers the tile)
    int wz;         // first weight block of the unit (K block 0); a stage adds 2 * ks
    int m0;         // GEMM2: first output feature of the unit
};

// Token tiles the GEMMs run over (generic pointers: global or shared memory).
struct TileView {
    const int* expert;
    const int* row0;
    const int* rows;
    int ntiles;
};

// Unit u -> (phase, tile, weight block), tile by tile: the units of one tile
// are consecutive, so the SMs that take them read that tile's token rows at
// about the same time.
__device__ __forceinline__ bool decode_unit(const GemmArgs& g, const TileView& tv, int u, Unit& un)
{
    const int nb1 = g.I / kTile;
    const int nb2 = (g.H + 2 * kTile - 1) / (2 * kTile);
    const int units1 = (g.phases & 1) ? tv.ntiles * nb1 : 0;
    const int units2 = (g.phases & 2) ? tv.ntiles * nb2 : 0;
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
    // (debug builds: a tile outside the experts or the reserved rows ends the
    // role's loop, like the end of the units, with the error latched)
    if (!MM_CHECK(un.expert >= 0 && un.expert < g.P && un.row0 >= 0 && un.rows >= 1 && un.rows <= 128 &&
                      un.row0 + un.rows <= g.rows_cap,
                  g.status, kSiteGemmTile))
        return false;
    un.tbox = un.rows <= 16 ? 0 : (un.rows <= 32 ? 1 : (un.rows <= 64 ? 2 : 3));
    if (un.phase == 1) {
        un.nw = 2;
        un.ksteps = g.H / kKStep;
        un.wz = (un.expert * nb1 + un.blk) * un.ksteps * 2;
        un.m0 = 0;
    } else {
        un.m0 = 2 * un.blk * kTile;
        un.nw = (un.m0 + kTile < g.H) ? 2 : 1;
        un.ksteps = g.I / kKStep;
        un.wz = (un.expert * nb2 + un.blk) * un.ksteps * 2;
    }
    return true;
}

__device__ __forceinline__ int ld_acquire(const int* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// shared-memory carve-up of the GEMM machinery (base aligned to 1024 bytes)
constexpr int kURing = 4;                // units queued ahead in shared memory
struct GemmSmem {
    uint8_t* stages;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tmem_full;
    uint64_t* tmem_empty;
    uint64_t* ufull;          // [kURing] unit slot written (producer)
    uint64_t* uempty;         // [kURing] unit slot read (MMA warp, weight-side producer, every epilogue thread)
    uint64_t* drain;          // the MMA thread's own wait for its issued work after an abort
    // CTA pairs (the 2-SM GEMM): the unit numbers CTA 0 draws reach CTA 1
    // through CTA 1's inbox; CTA 1 reports its drained accumulator to CTA 0,
    // which issues the pair's MMAs
    uint64_t* inbox_full;     // [kURing] in CTA 1: a number arrived
    uint64_t* inbox_free;     // [kURing] in CTA 0: CTA 1 took a number out
    uint64_t* peer_tmem_empty;  // in CTA 0: CTA 1's epilogue drained its accumulator
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    volatile int* uring;      // [kURing] unit numbers
    volatile int* inbox;      // [kURing] numbers drawn by CTA 0 (in CTA 1)
};
// Barrier block (kBarBlock bytes): full[8], empty[8], tmem_full, tmem_empty,
// ufull[4], uempty[4], drain, inbox_full[4], inbox_free[4],
// peer_tmem_empty, then the TMEM base, the abort flag, the unit ring and the
// inbox.  Its layout does not depend on the stage count, so one kernel can run
// either geometry over the same buffers.
constexpr int kMaxStages = 8;
__device__ __forceinline__ GemmSmem gemm_smem(uint8_t* stages, uint8_t* bars)
{
    GemmSmem s;
    s.stages = stages;
    s.full = reinterpret_cast<uint64_t*>(bars);
    s.empty = s.full + kMaxStages;
    s.tmem_full = s.empty + kMaxStages;
    s.tmem_empty = s.tmem_full + 1;
    s.ufull = s.tmem_empty + 1;
    s.uempty = s.ufull + kURing;
    s.drain = s.uempty + kURing;
    s.inbox_full = s.drain + 1;
    s.inbox_free = s.inbox_full + kURing;
    s.peer_tmem_empty = s.inbox_free + kURing;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.peer_tmem_empty + 1);
    s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
    s.uring = s.abort_flag + 1;
    s.inbox = s.uring + kURing;
    static_assert((2 * kMaxStages + 4 + 4 * kURing) * 8 + 8 + 8 * kURing <= kBarBlock, "barrier block");
    return s;
}

// All threads: barriers, tensor-memory allocation (warp 1); returns the TMEM
// base.  Both producer threads (token side and weight side) arrive on every
// full barrier; the weight side takes every unit out of the ring.
template <class G>
__device__ __forceinline__ uint32_t gemm_setup(const GemmSmem& s, const GemmMaps& maps)
{
    const int warp = threadIdx.x >> 5;
    constexpr uint32_t kProducers = 2;
    if (threadIdx.x == 0) {
        for (int i = 0; i < G::kStages; ++i) {
            mbar_init(&s.full[i], kProducers);
            mbar_init(&s.empty[i], 1);
        }
        mbar_init(s.tmem_full, 1);
        mbar_init(s.tmem_empty, kEpiThreads);
        mbar_init(s.drain, 1);
        for (int i = 0; i < kURing; ++i) {
            mbar_init(&s.ufull[i], 1);
            mbar_init(&s.uempty[i], kProducers + kEpiThreads);
        }
        *s.abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&maps.w1);
        prefetch_tmap(&maps.w2);
        prefetch_tmap(&maps.w2_one);
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

// ---- unit queue ----------------------------------------------------------------
struct UnitQueue {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance()
    {
        if (++slot == kURing) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// CTA pairs: CTA 0 draws the next number and hands it to CTA 1 through CTA
// 1's inbox (a remote store and a remote arrive); CTA 1 takes it out and
// frees the slot with a remote arrive on CTA 0's inbox_free.  Bounded waits.
__device__ __forceinline__ bool pair_draw(const GemmArgs& g, const GemmSmem& s, UnitQueue& box, uint32_t rank, int& u)
{
    if (rank == 0) {
        u = *s.abort_flag ? 0x7FFFFFFF : atomicAdd(g.unit_next, 1);
        if (!mbar_wait_cluster(&s.inbox_free[box.slot], box.phase ^ 1u, g.status, s.abort_flag, kSiteUnitQueue))
            return false;
        st_peer_u32(peer_addr(const_cast<int*>(&s.inbox[box.slot]), 1), static_cast<uint32_t>(u));
        mbar_arrive_peer(peer_addr(&s.inbox_full[box.slot], 1));
    } else {
        if (!mbar_wait_cluster(&s.inbox_full[box.slot], box.phase, g.status, s.abort_flag, kSiteUnitQueue))
            return false;
        u = s.inbox[box.slot];
        mbar_arrive_peer(peer_addr(&s.inbox_free[box.slot], 0));
    }
    box.advance();
    return true;
}

// Producer: take the next unit number (drawn here, or for the second CTA of a
// pair handed over by the first) and queue it for the CTA's consumers.
__device__ __forceinline__ bool push_unit(const GemmArgs& g, const GemmSmem& s, UnitQueue& q, int& u,
                                          UnitQueue* box = nullptr, uint32_t rank = 0)
{
    if (box) {
        if (!pair_draw(g, s, *box, rank, u)) return false;
    } else {
        u = *s.abort_flag ? 0x7FFFFFFF : atomicAdd(g.unit_next, 1);
    }
    if (!mbar_wait(&s.uempty[q.slot], q.phase ^ 1u, g.status, s.abort_flag, kSiteUnitQueue)) return false;
    s.uring[q.slot] = u;
    mbar_arrive(&s.ufull[q.slot]);
    q.advance();
    return true;
}

// MMA thread / epilogue thread: the next unit the producer queued.
__device__ __forceinline__ bool pop_unit(const GemmArgs& g, const GemmSmem& s, UnitQueue& q, int& u)
{
    if (!mbar_wait(&s.ufull[q.slot], q.phase, g.status, s.abort_flag, kSiteUnitQueue)) return false;
    u = s.uring[q.slot];
    mbar_arrive(&s.uempty[q.slot]);
    q.advance();
    return true;
}

// ---- producers ----------------------------------------------------------------
// kSideTokens: the token side (draws the units, waits for GEMM1 results before
// a GEMM2 unit); kSideWeights: the weight side (takes the units out of the
// ring like the consumers).
constexpr int kSideTokens = 1, kSideWeights = 2;

template <class G, int kSide>
__device__ __forceinline__ void producer_loop(const GemmMaps& maps, const GemmArgs& g, const TileView& tv,
                                              const GemmSmem& s)
{
    constexpr bool kTok = kSide == kSideTokens, kW = kSide == kSideWeights;
    const uint64_t pol_w = g.keep_weights ? policy_evict_normal() : policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    constexpr int kStages = G::kStages;
    int armed[kStages];
    for (int i = 0; i < kStages; ++i) armed[i] = -1;
    Unit un;
    UnitQueue q;
    for (;;) {
        int u;
        const bool got = kSide == kSideWeights ? pop_unit(g, s, q, u) : push_unit(g, s, q, u);
        if (!got || *s.abort_flag || !decode_unit(g, tv, u, un)) break;
        const CUtensorMap* wmap = un.phase == 1 ? &maps.w1 : (un.nw == 2 ? &maps.w2 : &maps.w2_one);
        const CUtensorMap* amap = un.phase == 1 ? &maps.xq[un.tbox] : &maps.hq[un.tbox];
        const uint8_t* wsf = un.phase == 1 ? g.w1_sf : g.w2_sf;
        const uint8_t* asf = un.phase == 1 ? g.xs_t : g.hs_t;
        if (kTok && un.phase == 2) {
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
        const uint32_t bytes = (kTok ? (kBBox << un.tbox) * kKStep + kSFBytes : 0) +
                               (kW ? un.nw * (kWBoxTxBytes + kSFBytes) : 0);
        const uint8_t* wblk = (un.phase == 1 ? g.w1 : g.w2) + static_cast<int64_t>(un.wz) * kWBoxTxBytes;
        if (kW && kPrefetch > 0) {
            // the first stages of the unit; later ones are requested kPrefetch stages ahead
            for (int j = 1; j < kPrefetch && j < un.ksteps; ++j)
                prefetch_l2(wblk + static_cast<int64_t>(2 * j) * kWBoxTxBytes, un.nw * kWBoxTxBytes);
        }
        for (int ks = 0; ks < un.ksteps; ++ks) {
            if (kW && kPrefetch > 0 && ks + kPrefetch < un.ksteps)
                prefetch_l2(wblk + static_cast<int64_t>(2 * (ks + kPrefetch)) * kWBoxTxBytes, un.nw * kWBoxTxBytes);
            if (!mbar_wait(&s.empty[stage], phase ^ 1u, g.status, s.abort_flag, kSiteProducerEmpty)) break;
            uint8_t* st = s.stages + stage * G::kStageBytes;
            uint8_t* sf = st + G::kABytes + 2 * kWBoxBytes;
            mbar_arrive_expect_tx(&s.full[stage], bytes);
            armed[stage] = static_cast<int>(phase);
            // four copies per stage: token rows, token scales, the weight block
            // pair, the pair's scales
            if (kTok) {
                tma_load_2d(st, amap, ks * kKStep, un.row0, &s.full[stage], pol_a);
                bulk_load(sf, asf + (static_cast<int64_t>(un.tile) * un.ksteps + ks) * kSFBytes, kSFBytes,
                          &s.full[stage]);
            }
            if (kW) {
                const int wz = un.wz + 2 * ks;
                tma_load_3d(st + G::kABytes, wmap, 0, 0, wz, &s.full[stage], pol_w);
                bulk_load(sf + kSFBytes, wsf + static_cast<int64_t>(wz) * kSFBytes, un.nw * kSFBytes, &s.full[stage]);
            }
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (*s.abort_flag) {
        // let copies already in flight land before the CTA exits.  (A stage
        // the other producer never armed does not complete although this
        // side's copies landed: one deadline for all stages.)
        const uint64_t t0 = globaltimer();
        for (int i = 0; i < kStages; ++i) {
            if (armed[i] < 0) continue;
            while (!mbar_try_wait(&s.full[i], static_cast<uint32_t>(armed[i])))
                if (globaltimer() - t0 > kWaitLimitNs / 4) break;
        }
    }
}

// ---- MMA issuer: warp 1, all lanes --------------------------------------------
// The whole warp runs the loop, so descriptors and addresses are computed
// warp-uniformly; one elected lane issues the tensor-core instructions (the
// issuing thread's own operand arithmetic otherwise sets the rate of small
// MMAs).  Descriptors are built once; a stage only adds its offset (the
// address field of a descriptor counts 16-byte units and every stage lies
// below 256 KB, so the add never carries out of that field).  The instruction
// descriptors of a unit are formed once per unit.
__device__ __forceinline__ bool elect_one()
{
    uint32_t p;
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, e;\n\t}"
        : "=r"(p));
    return p != 0;
}

template <class G>
__device__ __forceinline__ void mma_loop(const GemmArgs& g, const TileView& tv, const GemmSmem& s, uint32_t tmem)
{
    const uint64_t a_desc0 = desc_kmajor_sw128(s.stages);
    const uint64_t b_desc0 = desc_kmajor_sw128(s.stages + G::kABytes);
    const uint64_t sf_desc0 = desc_sf(s.stages + G::kABytes + 2 * kWBoxBytes);
    constexpr int kStages = G::kStages;
    static_assert(kKStep == 4 * 32, "four MMAs of K = 32 per stage");
    static_assert(kStages * G::kStageBytes + 1024 < (1 << 18), "descriptor address field");
    constexpr uint64_t kStageDesc = G::kStageBytes >> 4, kSfDesc = kSFBytes >> 4;
    static_assert(kColSF + kMaxStages * kSFSlotCols <= kTmemCols, "scale slots fit the allocation");
    const int lane = threadIdx.x & 31;
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool aborted = false;
    Unit un;
    UnitQueue q;
    for (;;) {
        // the unit (every lane reads it; lane 0 accounts for the warp)
        const bool got = mbar_wait(&s.ufull[q.slot], q.phase, g.status, s.abort_flag, kSiteUnitQueue);
        if (!__all_sync(0xFFFFFFFFu, got)) break;
        const int u = s.uring[q.slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.uempty[q.slot]);
        q.advance();
        if (*s.abort_flag || !decode_unit(g, tv, u, un)) break;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(s.tmem_empty, acc_phase ^ 1u, g.status, s.abort_flag,
                                               kSiteMmaTmemEmpty))) {
            aborted = true;
            break;
        }
        tc_fence_after();
        const uint32_t n = static_cast<uint32_t>(un.nw * kTile);
        const uint32_t id0 = idesc_e4m3_e2m1(n, 0), id1 = idesc_e4m3_e2m1(n, 1);
        const uint32_t id2 = idesc_e4m3_e2m1(n, 2), id3 = idesc_e4m3_e2m1(n, 3);
        const bool two = un.nw == 2;
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
                tc_cp_32x128b_x4(t_sfa, sd);
                tc_cp_32x128b_x4(t_sfb, sd + kSfDesc);
                if (two) tc_cp_32x128b_x4(t_sfb + 4, sd + 2 * kSfDesc);
                if (ks == 0)
                    mma_mxf8f6f4_c<false>(tmem, ad, bd, id0, t_sfa, t_sfb);
                else
                    mma_mxf8f6f4_c<true>(tmem, ad, bd, id0, t_sfa, t_sfb);
                mma_mxf8f6f4_c<true>(tmem, ad + 2, bd + 2, id1, t_sfa, t_sfb);
                mma_mxf8f6f4_c<true>(tmem, ad + 4, bd + 4, id2, t_sfa, t_sfb);
                mma_mxf8f6f4_c<true>(tmem, ad + 6, bd + 6, id3, t_sfa, t_sfb);
                tc_commit(&s.empty[stage]);
            }
            __syncwarp();
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (aborted || *s.abort_flag) break;
        if (elect_one()) tc_commit(s.tmem_full);
        __syncwarp();
        acc_phase ^= 1u;
    }
    if (*s.abort_flag) {
        // drain issued tensor-core work before the allocation is freed, on a
        // barrier of its own: completing tmem_full here could let some epilogue
        // threads through while others have already left on the abort flag
        if (elect_one()) {
            tc_commit(s.drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(s.drain, 0))
                if (globaltimer() - t0 > kWaitLimitNs / 4) break;
        }
        __syncwarp();
    }
}

// 16 consecutive accumulator columns of this warp's 32 rows
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    tmem_ld_32x32b_x16(taddr, r);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- epilogue: warps 2..9 ------------------------------------------------------
// Warp w reads TMEM lanes 32*(w % 4) .. +32 (token rows) and column half
// (w - 2) / 4 of the unit's columns.
// dec(u, un): the unit behind number u (false: none).  A unit whose tile is
// absent (rows 0: the second CTA of a pair whose expert had an odd number of
// tiles) is drained and released like any other, and writes nothing.
// empty_remote: 0 = release the drained accumulator on this CTA's tmem_empty
// (every epilogue thread arrives); otherwise the cluster address of the barrier
// to arrive on: the second CTA of a pair reports straight to the CTA that
// issues the pair's MMAs, one relaxed arrive per warp once all its lanes have
// waited for their tensor-memory loads (nothing else needs ordering).
__device__ __forceinline__ void release_acc(const GemmSmem& s, uint32_t empty_remote, int lane)
{
    if (empty_remote) {
        __syncwarp();
        if (lane == 0) mbar_arrive_peer_relaxed(empty_remote);
    } else {
        mbar_arrive(s.tmem_empty);
    }
}

template <class Dec>
__device__ __forceinline__ void epilogue_loop(const GemmArgs& g, const GemmSmem& s, uint32_t tmem, const Dec& dec,
                                              uint32_t empty_remote = 0)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;                       // TMEM lane quarter
    const int half = (warp - kEpiWarp0) >> 2;     // which half of the columns
    const int r = 32 * q + lane;                  // token row within the tile
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16);
    uint32_t acc_phase = 0;
    Unit un;
    UnitQueue uq;
    for (;;) {
        int u;
        if (!pop_unit(g, s, uq, u) || *s.abort_flag || !dec(u, un)) break;
        if (!mbar_wait(s.tmem_full, acc_phase, g.status, s.abort_flag, kSiteEpiTmemFull)) break;
        tc_fence_after();
        const bool active = 32 * q < un.rows;                       // warp-uniform
        const bool row_ok = r < un.rows;
        float v[128];                                              // 128 accumulator values of this row
        if (un.phase == 1) {
            // columns [half*64, +64) = gate, [128 + half*64, +64) = up
            if (active) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float t16[16];
                    ld16(lane_addr + half * 64 + 16 * c, t16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[16 * c + i] = t16[i];
                    ld16(lane_addr + kTile + half * 64 + 16 * c, t16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[64 + 16 * c + i] = t16[i];
                }
                tmem_ld_wait();
            }
            tc_fence_before();
            release_acc(s, empty_remote, lane);
            if (active && row_ok) {
                const int64_t row = un.row0 + r;
                const int col0 = un.blk * kTile + half * 64;            // first I-column of this half
                const int kchunks = g.I / kKStep;
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    float* h = v + 32 * blk;                               // h overwrites gate
                    float amax = 0.0f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float gv = h[i];
                        h[i] = gv / (1.0f + __expf(-gv)) * v[64 + 32 * blk + i];
                        amax = fmaxf(amax, fabsf(h[i]));
                    }
                    const int X = mx_e4m3_exponent(amax);
                    const float inv = exp2i(-X);
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint32_t wd = 0;
                        if (amax > 0.0f) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) wd |= e4m3_code(h[4 * i + j], inv) << (8 * j);
                        }
                        pk[i] = wd;
                    }
                    uint4* dst = reinterpret_cast<uint4*>(g.hq + row * g.I + col0 + 32 * blk);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    g.hs_t[act_sf_offset(un.tile, r, col0 / 32 + blk, kchunks)] = static_cast<uint8_t>(X + 127);
                }
            }
            // publish this unit's share of hq for the tile's GEMM2 units
            fence_proxy_async_global();
            __threadfence();
            epi_bar_sync();
            if (threadIdx.x == kEpiWarp0 * 32 && un.rows > 0) atomicAdd(&g.done1[un.tile], 1);
        } else {
            // columns [half*128, +128) of this unit's weight rows
            const bool cols = half < un.nw;
            if (active && cols) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float t16[16];
                    ld16(lane_addr + half * kTile + 16 * c, t16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[16 * c + i] = t16[i];
                }
                tmem_ld_wait();
            }
            tc_fence_before();
            release_acc(s, empty_remote, lane);
            if (active && cols && row_ok) {
                const int m0 = un.m0 + half * kTile;                                    // first output feature
                uint4* dst = reinterpret_cast<uint4*>(g.y + static_cast<int64_t>(un.row0 + r) * g.H + m0);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    uint32_t o[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * i + 2 * j], v[8 * i + 2 * j + 1]);
                        o[j] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
        acc_phase ^= 1u;
    }
}

// All threads (kThreads): each warp runs its role over the units the CTA's
// token-side producer draws.
template <class G>
__device__ __forceinline__ void gemm_roles(const GemmMaps& maps, const GemmArgs& g, const TileView& tv,
                                           const GemmSmem& s, uint32_t tmem)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        if (lane == 0) producer_loop<G, kSideTokens>(maps, g, tv, s);
    } else if (warp == kWProdWarp) {
        if (lane == 0) producer_loop<G, kSideWeights>(maps, g, tv, s);
    } else if (warp == 1) {
        mma_loop<G>(g, tv, s, tmem);
    } else {
        epilogue_loop(g, s, tmem, [&](int u, Unit& un) { return decode_unit(g, tv, u, un); });
    }
}

}  // namespace mm
