// mm_internal.h -- shared definitions of the fused MoE library: the handle,
// tile geometry, the scale-factor tile layout and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <vector>

#include "../../include/megamoe.h"

namespace mm {

// ---- tile geometry --------------------------------------------------------
// Both GEMMs put one token tile on the MMA's M side (e4m3; the MMA is always
// M = 128, rows past the tile are ignored) and 256 weight rows on its N side
// (e2m1), K in stages of 128: gate + up rows of 128 I-columns for GEMM1, 256
// output features for GEMM2.
// Every physical expert's dispatched rows form a segment that starts at a
// multiple of kSegAlign rows and is cut into token tiles (kTokTile rows on the
// large-input path, kSmallTile rows in the fused small-input kernel), so a
// tile never straddles two experts.
#ifndef MM_STAGES
#define MM_STAGES 4
#endif
#ifndef MM_SMALL_STAGES
#define MM_SMALL_STAGES 5
#endif
#ifndef MM_PREFETCH
#define MM_PREFETCH 2
#endif
constexpr int kTile = 128;       // weight rows per TMA box / weight row block
constexpr int kTokTile = 128;    // token rows per tile, large-input path
constexpr int kSmallTile = 64;   // token rows per tile, fused small-input kernel
constexpr int kSegAlign = 16;    // segment start alignment (rows)
constexpr int kKStep = 128;      // reduction elements per pipeline stage
constexpr int kBBox = 16;        // token rows per TMA box of the token operand
constexpr int kPrefetch = MM_PREFETCH;  // weight stages requested into L2 ahead of the TMA loads
constexpr int kChunkPairs = 1024;  // (token, slot) pairs per permute chunk
constexpr int kSmallMaxTokens = 512;  // largest batch the fused small-input kernel takes

// shared-memory stage: tokens (A) | weights (B, two 128-row boxes) | SF(A, B0, B1)
constexpr int kWBoxBytes = kTile * kKStep;           // e2m1 unpacked to 1 byte/element in smem
constexpr int kWBoxTxBytes = kTile * kKStep / 2;     // what the TMA counts: the packed global bytes
constexpr int kSFBytes = 512;                        // 128 rows x 4 scale bytes

// Weight blocks.  A weight block is 128 rows x 128 K of one expert.  Blocks
// are stored in GEMM-unit order: expert, group (the unit's pair of 128-row
// blocks), K block, then the pair's two members side by side, so one 3-D TMA
// box (z extent 2) and one 1 KB bulk copy fetch a unit's whole stage.
//   W1 (rows_per_expert = 2I): group = n-block nb, member 0 = the gate rows
//       [nb*128, +128), member 1 = the up rows [I + nb*128, +128);
//   W2 (rows_per_expert = H): group = m-block mb, members = rows
//       [mb*256, +128) and [mb*256 + 128, +128) (the second is absent when
//       H % 256 == 128 and mb is the last group).
struct WOrder {
    int rows_per_expert;
    int groups;       // groups per expert
    int kblocks;      // K / 128
    int gate_up;      // 1: W1 pairing, 0: W2 pairing
};

__host__ __device__ inline int64_t w_block(const WOrder& o, int64_t row, int kb)
{
    const int64_t p = row / o.rows_per_expert;
    const int lrb = static_cast<int>((row % o.rows_per_expert) / 128);
    int group, member;
    if (o.gate_up) {
        const int half_blocks = o.rows_per_expert / 256;
        group = lrb % half_blocks;
        member = lrb / half_blocks;
    } else {
        group = lrb / 2;
        member = lrb % 2;
    }
    return ((p * o.groups + group) * o.kblocks + kb) * 2 + member;
}

// Packed e2m1 bytes: each block is one contiguous 8 KB tile, rows of 64 bytes,
// so a TMA box reads sequential HBM.
__host__ __device__ inline int64_t w_tile_offset(const WOrder& o, int64_t row, int64_t byte_col)
{
    return w_block(o, row, static_cast<int>(byte_col / 64)) * 8192 + (row % 128) * 64 + (byte_col % 64);
}

// e8m0 scales: one 512-byte scale tile per block, in which row r, scale byte b
// (the 32-wide K block b of the block's 128) sits at (r%32)*16 + ((r%128)/32)*4
// + b -- the order in which tcgen05.cp 32x128b.warpx4 places scales in tensor
// memory for the block-scaled MMA (one 32-bit column per 32-row quarter).
__host__ __device__ inline int64_t w_sf_offset(const WOrder& o, int64_t row, int kblock32)
{
    return w_block(o, row, kblock32 / 4) * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4 + (kblock32 % 4);
}

inline WOrder w1_order(int H, int I) { return WOrder{2 * I, I / 128, H / 128, 1}; }
inline WOrder w2_order(int H, int I) { return WOrder{H, (H + 255) / 256, I / 128, 0}; }
inline int64_t w_blocks(const WOrder& o, int P) { return static_cast<int64_t>(P) * o.groups * o.kblocks * 2; }

// Activation scale tiles are per token tile: tile t, row r of the tile
// (r < 128), 32-element block b along K.
__host__ __device__ inline int64_t act_sf_offset(int64_t tile, int r, int kblock32, int kchunks)
{
    return (tile * kchunks + kblock32 / 4) * 512 + (r % 32) * 16 + (r / 32) * 4 + (kblock32 % 4);
}

__host__ __device__ inline int seg_rows(int cnt) { return (cnt + kSegAlign - 1) / kSegAlign * kSegAlign; }
__host__ __device__ inline int tiles_of(int cnt, int tile = kTokTile) { return (cnt + tile - 1) / tile; }

constexpr int kTokBoxes = 4;     // token-operand maps with boxes of 16, 32, 64, 128 rows

struct GemmMaps {
    CUtensorMap w1;            // W1 blocks, box = the unit's block pair (z extent 2)
    CUtensorMap w2;            // W2 blocks, box = block pair
    CUtensorMap w2_one;        // W2 blocks, box = one block (ragged last group; each CTA of a pair)
    CUtensorMap w1_one;        // W1 blocks, box = one block (each CTA of a pair)
    CUtensorMap w1_sf, w2_sf;  // weight scale tiles as rows of 256 bytes, box = a block pair's two tiles
    CUtensorMap xs_sf, hs_sf;  // token-tile scale tiles, box = one tile
    CUtensorMap xq[kTokBoxes]; // e4m3 [rows][H], box 16 << i rows
    CUtensorMap hq[kTokBoxes]; // e4m3 [rows][I], box 16 << i rows
};

// a16w4 GEMM (bf16 tokens): token maps over the dispatched bf16 rows and over
// h in bf16, boxes of 64 elements x (16 << i) rows.
struct Gemm16Maps {
    CUtensorMap xd[kTokBoxes];   // bf16 [rows][H]
    CUtensorMap hb[kTokBoxes];   // bf16 [rows][I]
};

struct Gemm16Args {
    const uint8_t* w1;
    const uint8_t* w1_sf;
    const uint8_t* w2;
    const uint8_t* w2_sf;
    __nv_bfloat16* hb;      // [rows][I]
    __nv_bfloat16* y;       // [rows][H]
    const int* tile_expert;
    const int* tile_row0;
    const int* tile_rows;
    const int* num_tiles;
    int* done1;
    int* unit_next;
    int* status;
    int H, I;
    int fault;
    int P, rows_cap;        // bounds checks of debug builds
};

struct GemmArgs {
    const uint8_t* w1;      // weight blocks in unit order (packed e2m1, 8 KB per block)
    const uint8_t* w2;
    const uint8_t* w1_sf;   // scale tiles, one 512-byte tile per W1 block
    const uint8_t* w2_sf;   // scale tiles, one per W2 block
    const uint8_t* xs_t;    // per token tile [tiles][H/128][512]
    uint8_t* hq;            // [rows][I]
    uint8_t* hs_t;          // per token tile [tiles][I/128][512]
    __nv_bfloat16* y;       // [rows][H]
    const int* tile_expert; // per token tile
    const int* tile_row0;
    const int* tile_rows;
    const int* num_tiles;
    int* done1;             // per token tile: GEMM1 units finished
    int* unit_next;         // next unit to hand out (zeroed before the GEMM phase)
    int* status;
    int H, I, P;
    int phases;             // bit 0: GEMM1 units, bit 1: GEMM2 units
    int fault;              // injected fault (FaultSite), 0 = none
    int rows_cap;           // dispatch rows reserved (bounds checks of debug builds)
    const int* st_tile;     // the 2-SM GEMM's tile pairs [2 * num_tiles[2]]
    int keep_weights;       // 1: weight loads with the normal L2 policy (an expert's tiles re-read its
                            // weights); 0: evict-first (streamed once, the fused small-input kernel)
    int select;             // 0: run; 1: run unless num_tiles[3] chose the pair kernel; 2: run only if it did
};

// The tile scan's choice between the large-input GEMM kernels (num_tiles[3]):
// the pair kernel gives each pair of an expert's tiles one M = 256 MMA, so an
// expert with an odd tile count costs it a whole extra tile of MMA work; it is
// chosen when those extra tiles are at most 1/64 of all tiles.
__host__ __device__ inline int choose_pairs(int tiles, int pairs) { return (2 * pairs - tiles) * 64 <= tiles ? 1 : 0; }

}  // namespace mm

struct mm_ctx {
    int dev = 0, sms = 0;
    int E = 0, P = 0, k = 0, H = 0, I = 0;
    int ns = 0;                     // fused shared experts (mm_set_shared_experts): physical P .. P+ns-1
    int small_max = 512, large_min = 1024;
    int route = MM_ROUTE_AUTO, layer = 0, recording = 0;
    int fault = 0;                  // mm::FaultSite
    // large-input GEMM kernel (MM_GEMM_2SM): 0 one CTA per unit, 1 CTA pairs
    // (2-SM MMAs) when the shapes allow, 2 chosen per batch on the device from
    // the tile counts (both kernels are launched; the one not chosen returns)
    int gemm_2sm = 2;
    // weights (library-owned)
    uint8_t *w1 = nullptr, *w1_sf = nullptr, *w2 = nullptr, *w2_sf = nullptr;
    bool weights_set = false;
    // EPLB map
    int32_t *map = nullptr, *rc = nullptr;
    int R = 1;
    std::vector<int32_t> host_map, host_rc;   // the installed map, host copy (rebalancing)
    bool map_set = false;
    // per-layer logical counts [MM_MAX_LAYERS][E]
    int64_t* counts = nullptr;
    // workspace
    int64_t cap_tokens = 0, rows_cap = 0, tiles_cap = 0, chunks_cap = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int32_t *idx = nullptr, *phys = nullptr, *pos = nullptr;
    float* wgt = nullptr;
    int32_t *chunk_hist = nullptr, *off = nullptr, *toff = nullptr, *tile_expert = nullptr, *tile_row0 = nullptr,
            *tile_rows = nullptr, *num_tiles = nullptr, *done1 = nullptr;
    int32_t* unit_next = nullptr;   // the GEMM kernels' unit counter (num_tiles[1])
    int32_t* st_tile = nullptr;     // tile pairs of the 2-SM GEMM [2 * tiles] (count in num_tiles[2])
    uint8_t *xq = nullptr, *xs_t = nullptr, *hq = nullptr, *hs_t = nullptr;
    __nv_bfloat16* y = nullptr;
    int* status = nullptr;
    unsigned* grid_bar = nullptr;   // fused kernel's grid barrier {count, generation}
    uint64_t* stamps = nullptr;     // fused kernel's per-CTA stage timestamps [sms][8]
    mm::GemmMaps maps{};
    mm::Gemm16Maps maps16{};
    int act = MM_ACT_MXFP8;          // activation format (mm_set_activation_format)
    int ws_act = MM_ACT_MXFP8;       // format the workspace was reserved for
    bool maps_weights = false, maps_ws = false;
    // per-launch timing of the dominant kernel: event pairs, pairs recorded so far
    std::vector<cudaEvent_t> prof_events;
    int prof_used = 0;
    // expert parallelism (mm_set_expert_parallel): this handle is rank ep_rank
    // of ep_world and holds the weights of physical experts
    // [ep_first[ep_rank], ep_first[ep_rank + 1]), ep_local of them
    bool ep = false;
    int ep_rank = 0, ep_world = 1, ep_local = 0;
    std::vector<int32_t> ep_first;     // [world + 1]
    int32_t* ep_local_id = nullptr;    // [P] device: index of each physical expert among its owner's
    int32_t* ep_recv_pos = nullptr;    // [ep_recv_cap] dispatch row of each received row
    int64_t ep_recv_cap = 0;
    int64_t ep_T = 0;                  // tokens of the last mm_ep_dispatch
    int64_t ep_send_rows = 0;          // send-buffer rows of the last mm_ep_dispatch
    // last forward (debug dumps)
    int last_route = 0, last_launches = 0, last_site = 0;
    int last_gemm = 0;              // grouped GEMM kernel of the last forward (stage 10 of mm_debug_dump)
    int64_t last_T = 0;
    cudaStream_t last_stream = nullptr;
};

namespace mm {

// sites of a device-side timeout (status[1])
enum WaitSite {
    kSiteProducerEmpty = 1,
    kSiteMmaFull = 2,
    kSiteMmaTmemEmpty = 3,
    kSiteEpiTmemFull = 4,
    kSiteProducerDone1 = 5,
    kSiteGridBarrier = 6,
    kSiteUnitQueue = 7,
    // sites of a failed device-side bounds check (debug builds, MM_ERR_DEVICE)
    kSiteRouteMap = 8,       // EPLB map entry or replica count outside its range
    kSitePermute = 9,        // a pair's physical expert outside [0, P) at the permute
    kSiteDispatch = 10,      // dispatch row or physical expert out of range at the quantise/dispatch copy
    kSiteGemmTile = 11,      // token tile with an expert or rows outside the reserved workspace
    kSiteCombine = 12,       // dispatch row outside the reserved rows at the combine
};

// Fault injection for the failure-detection tests (environment variable
// MM_FAULT, read at mm_create).  Each one only makes a bounded device-side wait
// unsatisfiable -- no invalid access, trap or endless loop -- so the wait must
// give up, latch MM_ERR_TIMEOUT with its site, and leave the context usable.
enum FaultSite {
    kFaultNone = 0,
    kFaultGridBarrier = 1,   // CTA 0 withholds its arrival at the fused kernel's second grid barrier
    kFaultGemmDependency = 2, // GEMM2 units wait for one GEMM1 unit more than a tile has
    // Debug builds only (MM_DEBUG): after mm_set_eplb_map has validated and
    // uploaded the map, one device map entry is overwritten with a physical id
    // past the last expert.  The route's bounds check must catch it before any
    // later stage indexes with it; a release build ignores this fault, since
    // without the checks the id would be used as an index.
    kFaultMapEntry = 3
};

// host-side launchers (return cudaGetLastError of the launch)
// slots per token (k routed + the shared experts) and physical experts of the
// routing (P routed + the shared experts)
inline int slots(const mm_ctx* c) { return c->k + c->ns; }
inline int pw(const mm_ctx* c) { return c->P + c->ns; }
// physical experts whose weights this handle holds: all of them, or under
// expert parallelism the rank's own range
inline int wexp(const mm_ctx* c) { return c->ep ? c->ep_local : c->P + c->ns; }

cudaError_t launch_route(const mm_ctx* c, const float* logits, const float* bias, int64_t T, cudaStream_t s);
cudaError_t launch_permute(const mm_ctx* c, int64_t T, cudaStream_t s);
// the same permute over any ids (negative ids left out) into pos
cudaError_t launch_permute_ids(const mm_ctx* c, const int32_t* ids, int64_t npairs, int P, int32_t* pos,
                               cudaStream_t s);
cudaError_t launch_quant_dispatch(const mm_ctx* c, const void* hidden, int64_t T, cudaStream_t s);
cudaError_t launch_gemm(const mm_ctx* c, int64_t T, cudaStream_t s);
cudaError_t launch_combine(const mm_ctx* c, void* out, int64_t T, cudaStream_t s);
cudaError_t launch_tile_scales(const uint8_t* src, uint8_t* dst, int64_t rows, int K, WOrder o, cudaStream_t s);
cudaError_t launch_tile_weights(const uint8_t* src, uint8_t* dst, int64_t rows, int K, WOrder o, cudaStream_t s);
cudaError_t gemm_prepare(int dev);
cudaError_t gemm2_prepare(int dev);
bool gemm2_usable(const mm_ctx* c);        // the large-input GEMM may run on CTA pairs for this handle
cudaError_t launch_gemm2(const mm_ctx* c, cudaStream_t s, int select);   // select: GemmArgs::select
// the large-input GEMM launch_gemm runs: 1 one CTA per unit, 2 CTA pairs, 4 chosen on the device (read
// num_tiles[3]: 0 one CTA, 1 pairs)
int gemm_kind(const mm_ctx* c);
cudaError_t gemm16_prepare();
cudaError_t launch_gemm16(const mm_ctx* c, cudaStream_t s);
cudaError_t launch_dispatch16(const mm_ctx* c, const void* hidden, int64_t T, cudaStream_t s);
cudaError_t small_prepare();
cudaError_t launch_small(const mm_ctx* c, const void* hidden, const float* logits, const float* bias, void* out,
                         int64_t T, cudaStream_t s);
void fill_gemm_args(const mm_ctx* c, GemmArgs* g);
mm_status reserve_pairs(mm_ctx* c, int64_t npairs, int64_t max_tokens);
void ep_release(mm_ctx* c);    // frees the expert-parallel buffers

}  // namespace mm
