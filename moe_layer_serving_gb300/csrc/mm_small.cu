// mm_small.cu -- the fused small-input kernel of the MoE forward (T <= 512):
// one cooperative launch, one CTA per SM, runs every stage of the layer
// (the pages' small-input path runs quantisation, dispatch, both expert GEMMs
// and the combine as a single kernel, "sglang PR #47065", Title/switches):
//
//   A  route + fused EPLB remap + count recording      (one warp per token)
//      -- grid barrier --
//   C  permute: every CTA rebuilds the expert segments, token tiles and the
//      stable dispatch rows in shared memory from the T*k physical ids
//   D  MXFP8 quantisation + dispatch copy               (one thread per block)
//      -- grid barrier --
//   F  GEMM1 (+SwiGLU, requant) and GEMM2 units, weight-streaming tcgen05
//      pipeline; a GEMM2 unit waits only for the GEMM1 units of its tile
//      -- grid barrier --
//   H  weighted combine                                  (one thread per 8 outputs)
//
// Every grid barrier and every wait is bounded; a timeout latches
// MM_ERR_TIMEOUT with its site, the remaining stages are skipped and the
// tensor memory is freed before the CTA exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mm_gemm.cuh"
#include "mm_stages.cuh"

namespace mm {
namespace {

// The GEMM phase's roles take kThreads threads (two producer warps, the MMA
// warp, eight epilogue warps); every other phase uses them all.
constexpr int kSmallThreads = kThreads;
constexpr int kSmallWarps = kSmallThreads / 32;
static_assert(kSmallThreads % 4 == 0, "quant_dispatch_block takes four consecutive lanes per K chunk");
constexpr int kMaxSmallPairs = kSmallMaxTokens * MM_MAX_TOPK;
// Two pipeline geometries over one buffer: short tiles with one more stage
// when every expert's rows fit in few short tiles (weight streaming, where the
// bytes in flight per SM set the rate), full tiles otherwise (fewer units,
// each expert's weights streamed fewer times).
constexpr int kStageRegion =
    GeomSmall::kStageRegion > GeomLarge::kStageRegion ? GeomSmall::kStageRegion : GeomLarge::kStageRegion;
constexpr int kMaxSmallTiles = MM_MAX_EXPERTS + kMaxSmallPairs / kSmallTile + 1;
constexpr int kSmallSmemBytes = kStageRegion + kBarBlock + 3 * kMaxSmallTiles * 4 + 64 + 1024;
static_assert(kSmallSmemBytes <= 232448, "shared memory per block");

struct SmallArgs {
    RouteArgs route;
    const __nv_bfloat16* x;   // hidden [T, H]
    __nv_bfloat16* out;       // [T, H]
    int32_t* pos;             // [T*k] dispatch rows (global copy)
    int32_t* off;             // [P+1]
    int32_t* tile_expert;     // global copies of the tile table (debug, combine)
    int32_t* tile_row0;
    int32_t* tile_rows;
    int32_t* num_tiles;
    uint8_t* xq;              // dispatched activation codes [rows, H]
    uint8_t* xs_t;            // their scale tiles
    unsigned* bar;            // grid barrier {count, generation}
    uint64_t* stamps;         // [gridDim.x][8] %globaltimer at the stage boundaries
    int P;
};

// Exclusive scan over the block's threads of three ints (every thread calls
// it): e[i] = the sum of v[i] over lower threads, t[i] = the block total.
// wsum: 99 ints of shared scratch.
constexpr int kScanVals = 3;
__device__ __forceinline__ void block_scan3(const int (&v)[kScanVals], int (&e)[kScanVals], int (&t)[kScanVals],
                                            int* wsum)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int in[kScanVals];
#pragma unroll
    for (int i = 0; i < kScanVals; ++i) in[i] = v[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int i = 0; i < kScanVals; ++i) {
            const int x = __shfl_up_sync(0xFFFFFFFFu, in[i], o);
            if (lane >= o) in[i] += x;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int i = 0; i < kScanVals; ++i) wsum[32 * i + warp] = in[i];
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < kScanVals; ++i) {
            const int x = lane < kSmallWarps ? wsum[32 * i + lane] : 0;
            int ix = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xFFFFFFFFu, ix, o);
                if (lane >= o) ix += u;
            }
            wsum[32 * i + lane] = ix - x;
            if (lane == 31) wsum[96 + i] = ix;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kScanVals; ++i) {
        e[i] = wsum[32 * i + warp] + in[i] - v[i];
        t[i] = wsum[96 + i];
    }
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Counting grid barrier over a 64-bit arrival count that only grows: every
// barrier adds exactly gridDim.x arrivals, so between barriers the count is a
// multiple of the grid, and a CTA whose arrival returned `old` waits (bounded)
// until the count reaches the next multiple above it.  The last CTA to arrive
// releases everyone with its own arrival: no reset, no second word.  (The host
// zeroes the count after a device error, when arrivals may be missing.)
__device__ bool grid_sync(unsigned* bar, int* status, volatile int* abort_flag, bool withhold = false)
{
    __syncthreads();
    if (threadIdx.x == 0 && !*abort_flag) {
        unsigned long long* cnt = reinterpret_cast<unsigned long long*>(bar);
        const unsigned long long G = gridDim.x;
        __threadfence();
        unsigned long long target;
        if (!withhold) {
            const unsigned long long old = atomicAdd(cnt, 1ull);
            target = old - old % G + G;
        } else {
            const unsigned long long cur = ld_acquire_u64(cnt);
            target = cur - cur % G + G;
        }
        const uint64_t t0 = globaltimer();
        while (ld_acquire_u64(cnt) < target) {
            if (globaltimer() - t0 > kWaitLimitNs) {
                latch_error(status, MM_ERR_TIMEOUT, kSiteGridBarrier);
                *abort_flag = 1;
                break;
            }
        }
        __threadfence();
    }
    __syncthreads();
    return !*abort_flag;
}

__global__ void __launch_bounds__(kSmallThreads, 1)
    small_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs g,
                 const __grid_constant__ SmallArgs a)
{
    // An error latched by an earlier launch and not yet read by the host may
    // have left the grid-barrier count short of a multiple of the grid: every
    // CTA then returns at once, doing no work and touching no barrier, and the
    // error stays latched for mm_get_status (which also resets the count).
    // Every CTA sees the same value here: within this launch nothing can
    // latch an error before a bounded wait has run out.
    if (*reinterpret_cast<volatile int*>(g.status) != 0) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const GemmSmem s = gemm_smem(smem, smem + kStageRegion);
    int* t_expert = reinterpret_cast<int*>(smem + kStageRegion + kBarBlock);
    int* t_row0 = t_expert + kMaxSmallTiles;
    int* t_rows = t_row0 + kMaxSmallTiles;
    int* scal = t_rows + kMaxSmallTiles;            // [0] tiles, [1] rows, [2] [3] tile counts
    static_assert(GeomSmall::kStages >= GeomLarge::kStages, "barriers initialised for the deeper pipeline");
    const uint32_t tmem = gemm_setup<GeomSmall>(s, maps);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t T = a.route.T;
    const int k = a.route.k + a.route.ns, P = a.P, H = g.H;     // slots per token, physical experts
    const int N = static_cast<int>(T) * k;
    const DispatchBounds chk{P, g.rows_cap, g.status};
    uint64_t* stamp = a.stamps + static_cast<int64_t>(blockIdx.x) * 8;
    if (threadIdx.x == 0) stamp[0] = globaltimer();

    // ---- A: route + EPLB remap + record ----------------------------------
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * kSmallWarps + warp; t < T;
         t += static_cast<int64_t>(gridDim.x) * kSmallWarps)
        route_token_any(a.route, t, lane, nullptr);

    if (threadIdx.x == 0) stamp[1] = globaltimer();
    bool ok = grid_sync(a.bar, g.status, s.abort_flag);
    if (threadIdx.x == 0) stamp[2] = globaltimer();

    // ---- C: permute, redundantly per CTA, in the (idle) pipeline buffers ----
    int* sphys = reinterpret_cast<int*>(s.stages);          // [N]
    int* spos = sphys + kMaxSmallPairs;                      // [N]
    int* wcnt = spos + kMaxSmallPairs;                       // [warps][P]: counts, then running bases
    int* cnt = wcnt + kSmallWarps * MM_MAX_EXPERTS;          // [P]
    int* soff = cnt + MM_MAX_EXPERTS;                        // [P+1]
    int* stoff = soff + MM_MAX_EXPERTS + 1;                  // [P]
    int* wsum = stoff + MM_MAX_EXPERTS;                      // [99] block-scan scratch
    static_assert((2 * kMaxSmallPairs + (kSmallWarps + 3) * MM_MAX_EXPERTS + 1 + 99) * 4 <= kStageRegion,
                  "permute scratch fits the pipeline buffers");
    const int chunk = ((N + kSmallWarps - 1) / kSmallWarps + 31) & ~31;
    bool short_tiles = true;
    const int lo = min(N, warp * chunk), hi = min(N, lo + chunk);
    const uint32_t lt = (1u << lane) - 1u;
    if (ok) {
        // the pairs' physical experts: each thread issues its loads before storing
        for (int i0 = threadIdx.x; i0 < N; i0 += 8 * kSmallThreads) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * kSmallThreads;
                v[u] = i < N ? a.route.phys[i] : 0;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * kSmallThreads;
                if (i < N) sphys[i] = v[u];
            }
        }
        for (int i = threadIdx.x; i < kSmallWarps * MM_MAX_EXPERTS; i += kSmallThreads) wcnt[i] = 0;
        __syncthreads();
        int* wc = wcnt + warp * MM_MAX_EXPERTS;
        for (int base = lo; base < hi; base += 32) {
            const int i = base + lane;
            const int p = i < hi ? sphys[i] : -1;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, p);
            if (p >= 0 && lane == __ffs(peers) - 1) wc[p] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        for (int p = threadIdx.x; p < P; p += kSmallThreads) {
            int run = 0;
            for (int w = 0; w < kSmallWarps; ++w) {
                const int v = wcnt[w * MM_MAX_EXPERTS + p];
                wcnt[w * MM_MAX_EXPERTS + p] = run;
                run += v;
            }
            cnt[p] = run;
        }
        __syncthreads();
        int tile;
        {
            // exclusive scans over experts of the padded segment sizes and of the
            // tile counts in both tile sizes (thread i takes experts [i * per,
            // i * per + per)); the totals choose the tile size: short tiles
            // unless they would add more than 1/16 to the tile count
            const int per = (P + kSmallThreads - 1) / kSmallThreads;
            const int p0 = min(P, static_cast<int>(threadIdx.x) * per), p1 = min(P, p0 + per);
            int v[kScanVals] = {0, 0, 0};
            for (int p = p0; p < p1; ++p) {
                v[0] += seg_rows(cnt[p]);
                v[1] += tiles_of(cnt[p], kSmallTile);
                v[2] += tiles_of(cnt[p], kTokTile);
            }
            int e[kScanVals], tot[kScanVals];
            block_scan3(v, e, tot, wsum);
            short_tiles = 16 * tot[1] <= 17 * tot[2];
            tile = short_tiles ? kSmallTile : kTokTile;
            int ro = e[0], to = short_tiles ? e[1] : e[2];
            for (int p = p0; p < p1; ++p) {
                soff[p] = ro;
                stoff[p] = to;
                ro += seg_rows(cnt[p]);
                to += tiles_of(cnt[p], tile);
            }
            if (threadIdx.x == 0) {
                soff[P] = tot[0];
                scal[0] = short_tiles ? tot[1] : tot[2];
                scal[1] = tot[0];
                scal[2] = tot[1];
                scal[3] = tot[2];
            }
        }
        __syncthreads();
        for (int p = threadIdx.x; p < P; p += kSmallThreads) {
            const int nt = tiles_of(cnt[p], tile);
            for (int t = 0; t < nt; ++t) {
                t_expert[stoff[p] + t] = p;
                t_row0[stoff[p] + t] = soff[p] + t * tile;
                t_rows[stoff[p] + t] = min(tile, cnt[p] - t * tile);
            }
        }
        for (int base = lo; base < hi; base += 32) {
            const int i = base + lane;
            const int p = i < hi ? sphys[i] : -1;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, p);
            int before = 0;
            if (p >= 0) {
                before = wc[p];
                spos[i] = soff[p] + before + __popc(peers & lt);
            }
            __syncwarp();
            if (p >= 0 && lane == __ffs(peers) - 1) wc[p] = before + __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        if (blockIdx.x == 0) {
            for (int i = threadIdx.x; i < N; i += kSmallThreads) a.pos[i] = spos[i];
            for (int p = threadIdx.x; p <= P; p += kSmallThreads) a.off[p] = soff[p];
            for (int t = threadIdx.x; t < scal[0]; t += kSmallThreads) {
                a.tile_expert[t] = t_expert[t];
                a.tile_row0[t] = t_row0[t];
                a.tile_rows[t] = t_rows[t];
                g.done1[t] = 0;
            }
            if (threadIdx.x == 0) {
                a.num_tiles[0] = scal[0];
                a.num_tiles[1] = 0;     // the GEMM phase's unit counter
            }
        }

        // ---- D: MXFP8 quantisation + dispatch ------------------------------
        const int nb = H / 32;
        for (int64_t it = static_cast<int64_t>(blockIdx.x) * kSmallThreads + threadIdx.x; it < T * nb;
             it += static_cast<int64_t>(gridDim.x) * kSmallThreads) {
            const int64_t t = it / nb;
            quant_dispatch_block(a.x, t, static_cast<int>(it % nb), H, k, spos + t * k, sphys + t * k, soff, stoff,
                                 tile, a.xq, a.xs_t, chk);
        }
        fence_proxy_async_global();
    }
    fence_proxy_async_shared();     // scratch writes above precede the TMA writes into the same buffers
    if (threadIdx.x == 0) stamp[3] = globaltimer();
    ok = grid_sync(a.bar, g.status, s.abort_flag, g.fault == kFaultGridBarrier && blockIdx.x == 0);
    if (threadIdx.x == 0) stamp[4] = globaltimer();

    // ---- F: GEMM1 + SwiGLU + requant, GEMM2 (tiles from shared memory) -----
    if (ok) {
        TileView tv;
        tv.expert = t_expert;
        tv.row0 = t_row0;
        tv.rows = t_rows;
        tv.ntiles = scal[0];
        if (short_tiles)
            gemm_roles<GeomSmall>(maps, g, tv, s, tmem);
        else
            gemm_roles<GeomLarge>(maps, g, tv, s, tmem);
    }
    gemm_teardown(tmem);
    if (threadIdx.x == 0) stamp[5] = globaltimer();
    ok = grid_sync(a.bar, g.status, s.abort_flag);
    if (threadIdx.x == 0) stamp[6] = globaltimer();

    // ---- H: combine ---------------------------------------------------------
    if (ok) {
        const int nc = H / 8;
        for (int64_t it = static_cast<int64_t>(blockIdx.x) * kSmallThreads + threadIdx.x; it < T * nc;
             it += static_cast<int64_t>(gridDim.x) * kSmallThreads)
            combine_chunk(g.y, a.route.w, a.pos, it / nc, static_cast<int>(it % nc), H, k, a.out, chk);
    }
    __syncthreads();
    if (threadIdx.x == 0) stamp[7] = globaltimer();
}

}  // namespace
}  // namespace mm

namespace mm {

cudaError_t small_prepare()
{
    return cudaFuncSetAttribute(small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallSmemBytes);
}

cudaError_t launch_small(const mm_ctx* c, const void* hidden, const float* logits, const float* bias, void* out,
                         int64_t T, cudaStream_t s)
{
    GemmArgs g;
    fill_gemm_args(c, &g);
    SmallArgs a;
    a.route.logits = logits;
    a.route.bias = bias;
    a.route.map = c->map;
    a.route.rc = c->rc;
    a.route.idx = c->idx;
    a.route.w = c->wgt;
    a.route.phys = c->phys;
    a.route.counts = c->recording ? c->counts + static_cast<int64_t>(c->layer) * c->E : nullptr;
    a.route.T = T;
    a.route.E = c->E;
    a.route.k = c->k;
    a.route.ns = c->ns;
    a.route.P = c->P;
    a.route.R = c->R;
    a.route.status = c->status;
    a.x = static_cast<const __nv_bfloat16*>(hidden);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.pos = c->pos;
    a.off = c->off;
    a.tile_expert = c->tile_expert;
    a.tile_row0 = c->tile_row0;
    a.tile_rows = c->tile_rows;
    a.num_tiles = c->num_tiles;
    a.xq = c->xq;
    a.xs_t = c->xs_t;
    a.bar = c->grid_bar;
    a.stamps = c->stamps;
    a.P = pw(c);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c->sms));
    cfg.blockDim = dim3(kSmallThreads);
    cfg.dynamicSmemBytes = kSmallSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, small_kernel, c->maps, g, a);
}

}  // namespace mm
