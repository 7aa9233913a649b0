// mm_route.cu -- the SIMT stages of the fused MoE forward on sm_103a:
//   router (sigmoid top-k) + fused EPLB remap + per-expert load recording,
//   the stable permute into expert-sorted segments (16-row aligned),
//   MXFP8 activation quantisation fused with the dispatch copy,
//   the deterministic gather combine,
//   and the re-layout of e8m0 scales into scale tiles (weights, at load time).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mm_device.cuh"
#include "mm_internal.h"
#include "mm_stages.cuh"

namespace mm {
namespace {

constexpr int kRouteWarps = 8;

// One warp per token; selections counted in shared memory, then once per CTA
// into the bound layer's global count table.
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(RouteArgs a)
{
    __shared__ int hist[MM_MAX_EXPERTS];
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + (threadIdx.x >> 5);
    if (t < a.T) route_token_any(a, t, threadIdx.x & 31, hist);
    if (a.counts) {
        __syncthreads();
        for (int e = threadIdx.x; e < a.E; e += blockDim.x)
            if (hist[e]) atomicAdd(reinterpret_cast<unsigned long long*>(a.counts + e),
                                   static_cast<unsigned long long>(hist[e]));
    }
}

// ---------------------------------------------------------------------------
// permute: chunk histograms -> per-expert scan (segments padded to 16 rows,
// token tiles of up to 128 rows) -> stable scatter (pairs keep (token, slot) order)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) hist_kernel(const int32_t* phys, int64_t npairs, int P, int32_t* chunk_hist,
                                                   int* status)
{
    (void)status;
    __shared__ int hist[MM_MAX_EXPERTS];
    for (int p = threadIdx.x; p < P; p += blockDim.x) hist[p] = 0;
    __syncthreads();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kChunkPairs;
    for (int i = threadIdx.x; i < kChunkPairs; i += blockDim.x) {
        const int64_t g = base + i;
        if (g < npairs) {
            // a negative id is a row to leave out (a padding row received
            // from another rank); ids at or past P are errors
            const int p = phys[g];
            if (p >= 0 && MM_CHECK(p < P, status, kSitePermute)) atomicAdd(&hist[p], 1);
        }
    }
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) chunk_hist[static_cast<int64_t>(blockIdx.x) * P + p] = hist[p];
}

// inclusive block scan of one int per thread (blockDim.x = 512)
__device__ int block_scan_incl(int v, int* warp_tot)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) warp_tot[w] = v;
    __syncthreads();
    if (w == 0) {
        int x = lane < (blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, x, off);
            if (lane >= off) x += o;
        }
        warp_tot[lane] = x;
    }
    __syncthreads();
    const int add = w > 0 ? warp_tot[w - 1] : 0;
    __syncthreads();
    return v + add;
}

struct ScanArgs {
    int32_t* chunk_hist;   // in: counts per chunk; out: exclusive base per chunk
    int nchunks, P;
    int32_t* off;          // [P+1] padded segment starts
    int32_t* toff;         // [P] first token tile of each expert
    int32_t* tile_expert;
    int32_t* tile_row0;
    int32_t* tile_rows;
    int32_t* num_tiles;    // [0] tiles; [1] the GEMM kernel's unit counter, reset here; [2] tile pairs
    int32_t* done1;
    int32_t* st_tile;      // [2 * pairs]: the two tiles of each pair of an expert's tiles (second -1 if none)
};

__global__ void __launch_bounds__(512) scan_kernel(ScanArgs a)
{
    __shared__ int warp_tot[32];
    const int p = threadIdx.x;
    int cnt = 0;
    if (p < a.P) {
        // exclusive prefix over the chunks of this expert's counts; each batch
        // of loads is issued before its stores
        constexpr int kBatch = 16;
        int32_t* h = a.chunk_hist + p;
        for (int c0 = 0; c0 < a.nchunks; c0 += kBatch) {
            int v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                v[u] = c0 + u < a.nchunks ? h[static_cast<int64_t>(c0 + u) * a.P] : 0;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (c0 + u < a.nchunks) h[static_cast<int64_t>(c0 + u) * a.P] = cnt;
                cnt += v[u];
            }
        }
    }
    const int padded = seg_rows(cnt);
    const int tiles = tiles_of(cnt);
    const int pairs = (tiles + 1) / 2;
    const int off_incl = block_scan_incl(padded, warp_tot);
    const int tiles_incl = block_scan_incl(tiles, warp_tot);
    const int pairs_incl = block_scan_incl(pairs, warp_tot);
    if (p < a.P) {
        const int off = off_incl - padded;
        const int t0 = tiles_incl - tiles;
        const int s0 = pairs_incl - pairs;
        a.off[p] = off;
        a.toff[p] = t0;
        for (int t = 0; t < tiles; ++t) {
            a.tile_expert[t0 + t] = p;
            a.tile_row0[t0 + t] = off + t * kTokTile;
            a.tile_rows[t0 + t] = min(kTokTile, cnt - t * kTokTile);
            a.done1[t0 + t] = 0;
        }
        // the expert's tiles two by two, for the GEMM on CTA pairs
        for (int i = 0; i < pairs; ++i) {
            a.st_tile[2 * (s0 + i)] = t0 + 2 * i;
            a.st_tile[2 * (s0 + i) + 1] = 2 * i + 1 < tiles ? t0 + 2 * i + 1 : -1;
        }
        if (p == a.P - 1) {
            a.off[a.P] = off_incl;
            a.num_tiles[0] = tiles_incl;
            a.num_tiles[1] = 0;
            a.num_tiles[2] = pairs_incl;
            a.num_tiles[3] = choose_pairs(tiles_incl, pairs_incl);
        }
    }
}

// Stable scatter of one chunk of (token, slot) pairs: eight warps take 128
// consecutive pairs each, count them per expert, take exclusive prefixes of
// those counts across warps (so a warp's pairs follow every earlier warp's in
// each expert's segment), then place their pairs in order.
constexpr int kScatterWarps = 8;
static_assert(kChunkPairs % (32 * kScatterWarps) == 0, "a chunk splits evenly over the warps");

// (Debug builds: a physical id outside [0, P) -- already reported by the
// histogram -- is left out like a pair past the end.)
__device__ __forceinline__ int scatter_id(const int32_t* phys, int64_t i, int64_t npairs, int P)
{
    int p = i < npairs ? phys[i] : -1;
#ifdef MM_DEBUG
    if (p >= P) p = -1;
#endif
    (void)P;
    return p;
}

__global__ void __launch_bounds__(32 * kScatterWarps) scatter_kernel(const int32_t* phys, int64_t npairs, int P,
                                                                     const int32_t* chunk_base, const int32_t* off,
                                                                     int32_t* pos)
{
    __shared__ int wcnt[kScatterWarps][MM_MAX_EXPERTS];   // per-warp counts, then the warp's bases
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    constexpr int kPer = kChunkPairs / kScatterWarps;
    for (int i = threadIdx.x; i < kScatterWarps * MM_MAX_EXPERTS; i += blockDim.x) (&wcnt[0][0])[i] = 0;
    __syncthreads();
    const int64_t base = static_cast<int64_t>(blockIdx.x) * kChunkPairs + w * kPer;
    const uint32_t lt = (1u << lane) - 1u;
    for (int it = 0; it < kPer / 32; ++it) {
        const int64_t i = base + it * 32 + lane;
        const int p = scatter_id(phys, i, npairs, P);
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, p);
        if (p >= 0 && lane == __ffs(peers) - 1) wcnt[w][p] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    const int32_t* cb = chunk_base + static_cast<int64_t>(blockIdx.x) * P;
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        int run = off[p] + cb[p];
        for (int x = 0; x < kScatterWarps; ++x) {
            const int v = wcnt[x][p];
            wcnt[x][p] = run;
            run += v;
        }
    }
    __syncthreads();
    for (int it = 0; it < kPer / 32; ++it) {
        const int64_t i = base + it * 32 + lane;
        const int p = scatter_id(phys, i, npairs, P);
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, p);
        int before = 0;
        if (p >= 0) {
            before = wcnt[w][p];
            pos[i] = before + __popc(peers & lt);
        }
        __syncwarp();
        if (p >= 0 && lane == __ffs(peers) - 1) wcnt[w][p] = before + __popc(peers);
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// MXFP8 quantisation + dispatch: one thread per 32-element block of a token;
// 4 x 128-bit loads, one e8m0 scale, 32 e4m3 codes written to each of the
// token's k dispatch rows (2 x 128-bit stores each).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_dispatch_kernel(const __nv_bfloat16* __restrict__ x, int64_t T, int H,
                                                            int k, const int32_t* __restrict__ pos,
                                                            const int32_t* __restrict__ phys,
                                                            const int32_t* __restrict__ off,
                                                            const int32_t* __restrict__ toff,
                                                            uint8_t* __restrict__ xq, uint8_t* __restrict__ xs_t,
                                                            DispatchBounds chk)
{
    const int nb = H / 32;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t t = g / nb;
    if (t >= T) return;
    quant_dispatch_block(x, t, static_cast<int>(g % nb), H, k, pos + t * k, phys + t * k, off, toff, kTokTile, xq,
                         xs_t, chk);
}

// a16w4 dispatch: token t's bf16 row copied to its k dispatch rows; one thread
// per 16-byte chunk (one load, k stores).
__global__ void __launch_bounds__(256) dispatch16_kernel(const uint4* __restrict__ x, int64_t T, int H, int k,
                                                         const int32_t* __restrict__ pos, uint4* __restrict__ xd,
                                                         DispatchBounds chk)
{
    const int nc = H / 8;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t t = g / nc;
    if (t >= T) return;
    const int c = static_cast<int>(g % nc);
    const uint4 v = x[t * nc + c];
    for (int j = 0; j < k; ++j) {
        const int64_t row = pos[t * k + j];
        if (MM_CHECK(row >= 0 && row < chk.rows_cap, chk.status, kSiteDispatch)) xd[row * nc + c] = v;
    }
}

// ---------------------------------------------------------------------------
// combine: out[t] = bf16( sum_j w[t,j] * y[pos[t,j]] ), fp32, j in order; one
// thread per 8 outputs (128-bit loads and stores), no atomics.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ y, const float* __restrict__ w,
                                                     const int32_t* __restrict__ pos, int64_t T, int H, int k,
                                                     __nv_bfloat16* __restrict__ out, DispatchBounds chk)
{
    const int nc = H / 8;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t t = g / nc;
    if (t >= T) return;
    combine_chunk(y, w, pos, t, static_cast<int>(g % nc), H, k, out, chk);
}

__global__ void tile_scales_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t rows, int K,
                                   WOrder o)
{
    const int nb = K / 32;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (g >= rows * nb) return;
    const int64_t r = g / nb;
    const int b = static_cast<int>(g % nb);
    dst[w_sf_offset(o, r, b)] = src[g];
}

// packed e2m1 [rows][K/2] -> 8 KB weight tiles, 16 bytes per thread
__global__ void tile_weights_kernel(const uint4* __restrict__ src, uint8_t* __restrict__ dst, int64_t rows, int K,
                                    WOrder o)
{
    const int per_row = K / 32;                    // 16-byte pieces per row
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (g >= rows * per_row) return;
    const int64_t r = g / per_row;
    const int c = static_cast<int>(g % per_row) * 16;
    *reinterpret_cast<uint4*>(dst + w_tile_offset(o, r, c)) = src[g];
}

unsigned grid_for(int64_t threads, int block) { return static_cast<unsigned>((threads + block - 1) / block); }

DispatchBounds bounds_of(const mm_ctx* c) { return DispatchBounds{pw(c), c->rows_cap, c->status}; }

}  // namespace

cudaError_t launch_route(const mm_ctx* c, const float* logits, const float* bias, int64_t T, cudaStream_t s)
{
    RouteArgs a;
    a.logits = logits;
    a.bias = bias;
    a.map = c->map;
    a.rc = c->rc;
    a.idx = c->idx;
    a.w = c->wgt;
    a.phys = c->phys;
    a.counts = c->recording ? c->counts + static_cast<int64_t>(c->layer) * c->E : nullptr;
    a.T = T;
    a.E = c->E;
    a.k = c->k;
    a.R = c->R;
    a.ns = c->ns;
    a.P = c->P;
    a.status = c->status;
    route_kernel<<<grid_for(T, kRouteWarps), kRouteWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_permute(const mm_ctx* c, int64_t T, cudaStream_t s)
{
    return launch_permute_ids(c, c->phys, T * slots(c), pw(c), c->pos, s);
}

cudaError_t launch_permute_ids(const mm_ctx* c, const int32_t* ids, int64_t npairs, int P, int32_t* pos,
                               cudaStream_t s)
{
    const int nchunks = static_cast<int>((npairs + kChunkPairs - 1) / kChunkPairs);
    hist_kernel<<<nchunks, 256, 0, s>>>(ids, npairs, P, c->chunk_hist, c->status);
    ScanArgs a;
    a.chunk_hist = c->chunk_hist;
    a.nchunks = nchunks;
    a.P = P;
    a.off = c->off;
    a.toff = c->toff;
    a.tile_expert = c->tile_expert;
    a.tile_row0 = c->tile_row0;
    a.tile_rows = c->tile_rows;
    a.num_tiles = c->num_tiles;
    a.done1 = c->done1;
    a.st_tile = c->st_tile;
    scan_kernel<<<1, 512, 0, s>>>(a);
    scatter_kernel<<<nchunks, 32 * kScatterWarps, 0, s>>>(ids, npairs, P, c->chunk_hist, c->off, pos);
    return cudaGetLastError();
}

cudaError_t launch_quant_dispatch(const mm_ctx* c, const void* hidden, int64_t T, cudaStream_t s)
{
    const int64_t threads = T * (c->H / 32);
    quant_dispatch_kernel<<<grid_for(threads, 256), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(hidden), T, c->H,
                                                                 slots(c), c->pos, c->phys, c->off, c->toff, c->xq,
                                                                 c->xs_t, bounds_of(c));
    return cudaGetLastError();
}

cudaError_t launch_dispatch16(const mm_ctx* c, const void* hidden, int64_t T, cudaStream_t s)
{
    const int64_t threads = T * (c->H / 8);
    dispatch16_kernel<<<grid_for(threads, 256), 256, 0, s>>>(static_cast<const uint4*>(hidden), T, c->H, slots(c),
                                                             c->pos, reinterpret_cast<uint4*>(c->xq), bounds_of(c));
    return cudaGetLastError();
}

cudaError_t launch_combine(const mm_ctx* c, void* out, int64_t T, cudaStream_t s)
{
    const int64_t threads = T * (c->H / 8);
    combine_kernel<<<grid_for(threads, 256), 256, 0, s>>>(c->y, c->wgt, c->pos, T, c->H, slots(c),
                                                          static_cast<__nv_bfloat16*>(out), bounds_of(c));
    return cudaGetLastError();
}

cudaError_t launch_tile_weights(const uint8_t* src, uint8_t* dst, int64_t rows, int K, WOrder o, cudaStream_t s)
{
    const int64_t threads = rows * (K / 32);
    tile_weights_kernel<<<grid_for(threads, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(src), dst, rows, K, o);
    return cudaGetLastError();
}

cudaError_t launch_tile_scales(const uint8_t* src, uint8_t* dst, int64_t rows, int K, WOrder o, cudaStream_t s)
{
    const int64_t threads = rows * (K / 32);
    tile_scales_kernel<<<grid_for(threads, 256), 256, 0, s>>>(src, dst, rows, K, o);
    return cudaGetLastError();
}

}  // namespace mm
