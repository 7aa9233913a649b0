// mm_api.cu -- the C ABI of the fused MoE layer: argument checks, owned
// device memory (weights, EPLB map, per-layer counts, workspace), TMA
// descriptors, route choice and the launch sequence of one forward.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "mm_internal.h"

using mm::kTile;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D row-major [rows][cols] tensor map, box [box_rows][box_cols elements]
// (128 bytes of them), 128-byte swizzle.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, void* base, uint64_t cols, uint64_t rows,
              uint64_t row_bytes, uint32_t box_rows, uint32_t box_cols = 128)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale tiles [n][512 bytes] read by TMA: rows of 256 bytes, a box of
// `box_rows` rows (2 = one tile, 4 = a block pair's two tiles), no swizzle, so
// shared memory receives the bytes as they are.
bool make_sf_map(CUtensorMap* m, void* base, uint64_t ntiles, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {256, 2 * ntiles};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {256, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weight blocks [nblocks][128 rows][128 e2m1]; a box is `depth` consecutive
// blocks (a GEMM unit's pair, or one block).
bool make_weight_map(CUtensorMap* m, void* base, uint64_t nblocks, uint32_t depth)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, 128, nblocks};
    const cuuint64_t strides[2] = {64, 8192};
    const cuuint32_t box[3] = {128, 128, depth};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int env_int(const char* name, int dflt)
{
    const char* v = getenv(name);
    if (!v || !*v) return dflt;
    char* end = nullptr;
    long x = strtol(v, &end, 10);
    return (end && *end == 0 && x >= 0 && x < (1L << 30)) ? static_cast<int>(x) : dflt;
}

#define CK(call)                                   \
    do {                                           \
        if ((call) != cudaSuccess) {               \
            cudaGetLastError();                    \
            return MM_ERR_CUDA;                    \
        }                                          \
    } while (0)

bool capturing(cudaStream_t s)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return st != cudaStreamCaptureStatusNone;
}

template <typename T>
T* carve(uint8_t*& p, size_t n)
{
    T* r = reinterpret_cast<T*>(p);
    p += (n * sizeof(T) + 255) & ~size_t(255);
    return r;
}

void free_ws(mm_ctx* c)
{
    if (c->ws) cudaFree(c->ws);
    c->ws = nullptr;
    c->ws_bytes = 0;
    c->cap_tokens = 0;
    c->maps_ws = false;
}

void profile_free(mm_ctx* c)
{
    for (cudaEvent_t e : c->prof_events)
        if (e) cudaEventDestroy(e);
    c->prof_events.clear();
    c->prof_used = 0;
}

}  // namespace

extern "C" {

const char* mm_status_string(mm_status s)
{
    switch (s) {
        case MM_OK: return "ok";
        case MM_ERR_INVALID_ARG: return "invalid argument";
        case MM_ERR_UNSUPPORTED: return "unsupported shape or device";
        case MM_ERR_NOT_READY: return "weights or EPLB map not set";
        case MM_ERR_CAPACITY: return "token count above capacity";
        case MM_ERR_CUDA: return "CUDA runtime error";
        case MM_ERR_TIMEOUT: return "device-side wait timed out";
        case MM_ERR_DEVICE: return "device-side check failed";
    }
    return "unknown status";
}

mm_status mm_create(int E, int P, int k, int H, int I, mm_handle* out)
{
    if (!out) return MM_ERR_INVALID_ARG;
    *out = nullptr;
    if (E < 1 || P < E || k < 1 || k > MM_MAX_TOPK || k > E || E > MM_MAX_EXPERTS || P > MM_MAX_EXPERTS ||
        H < 128 || I < 128 || H % 128 || I % 128 || H > 16384 || I > 8192)
        return MM_ERR_UNSUPPORTED;
    int dev = 0;
    CK(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    CK(cudaGetDeviceProperties(&prop, dev));
    if (prop.major != 10 || prop.minor != 3) return MM_ERR_UNSUPPORTED;
    if (!encode_fn()) return MM_ERR_UNSUPPORTED;
    mm_ctx* c = new (std::nothrow) mm_ctx();
    if (!c) return MM_ERR_CUDA;
    c->dev = dev;
    c->sms = prop.multiProcessorCount;
    c->E = E;
    c->P = P;
    c->k = k;
    c->H = H;
    c->I = I;
    {
        const char* f = getenv("MM_FAULT");
        if (f && !strcmp(f, "grid_barrier")) c->fault = mm::kFaultGridBarrier;
        else if (f && !strcmp(f, "gemm_dependency")) c->fault = mm::kFaultGemmDependency;
#ifdef MM_DEBUG
        else if (f && !strcmp(f, "map_entry")) c->fault = mm::kFaultMapEntry;
#endif
    }
    c->small_max = env_int("MM_SMALL_M_MAX", mm::kSmallMaxTokens);
    if (c->small_max > mm::kSmallMaxTokens) c->small_max = mm::kSmallMaxTokens;
    c->large_min = env_int("MM_LARGE_M_MIN", 1024);
    c->gemm_2sm = env_int("MM_GEMM_2SM", 2);        // 0 one CTA, 1 CTA pairs, 2 chosen per batch
    if (c->gemm_2sm < 0 || c->gemm_2sm > 2) c->gemm_2sm = 2;
    if (mm::gemm_prepare(dev) != cudaSuccess || mm::gemm2_prepare(dev) != cudaSuccess ||
        mm::small_prepare() != cudaSuccess ||
        mm::gemm16_prepare() != cudaSuccess ||
        cudaMalloc(&c->counts, sizeof(int64_t) * MM_MAX_LAYERS * E) != cudaSuccess ||
        cudaMemset(c->counts, 0, sizeof(int64_t) * MM_MAX_LAYERS * E) != cudaSuccess ||
        cudaMalloc(&c->status, 2 * sizeof(int)) != cudaSuccess ||
        cudaMemset(c->status, 0, 2 * sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        mm_destroy(c);
        return MM_ERR_CUDA;
    }
    if (P == E) {
        std::vector<int32_t> m(E), rc(E, 1);
        for (int e = 0; e < E; ++e) m[e] = e;
        mm_status st = mm_set_eplb_map(c, m.data(), rc.data(), 1);
        if (st != MM_OK) {
            mm_destroy(c);
            return st;
        }
    }
    *out = c;
    return MM_OK;
}

mm_status mm_destroy(mm_handle c)
{
    if (!c) return MM_OK;
    cudaDeviceSynchronize();
    cudaGetLastError();
    free_ws(c);
    profile_free(c);
    mm::ep_release(c);
    void* ptrs[] = {c->w1, c->w1_sf, c->w2, c->w2_sf, c->map, c->rc, c->counts, c->status};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    delete c;
    return MM_OK;
}

mm_status mm_set_weights(mm_handle c, const uint8_t* w1, const uint8_t* w1s, const uint8_t* w2, const uint8_t* w2s)
{
    if (!c || !w1 || !w1s || !w2 || !w2s) return MM_ERR_INVALID_ARG;
    if (!aligned(w1, 32) || !aligned(w2, 32) || !aligned(w1s, 16) || !aligned(w2s, 16)) return MM_ERR_INVALID_ARG;
    if (capturing(nullptr)) return MM_ERR_INVALID_ARG;
    const size_t P = mm::wexp(c), H = c->H, I = c->I;    // the physical experts this handle holds
    const mm::WOrder o1 = mm::w1_order(c->H, c->I), o2 = mm::w2_order(c->H, c->I);
    const size_t b1 = mm::w_blocks(o1, static_cast<int>(P)), b2 = mm::w_blocks(o2, static_cast<int>(P));
    const size_t n_w1 = b1 * 8192, n_w1s = b1 * 512;
    const size_t n_w2 = b2 * 8192, n_w2s = b2 * 512;
    if (!c->w1 || !c->w1_sf || !c->w2 || !c->w2_sf) {
        // all four buffers or none: a failed allocation frees the others, so a
        // later call never finds a partial set and writes through a null one
        uint8_t* buf[4] = {c->w1, c->w1_sf, c->w2, c->w2_sf};
        const size_t n[4] = {n_w1, n_w1s, n_w2, n_w2s};
        bool ok = true;
        for (int i = 0; i < 4 && ok; ++i)
            if (!buf[i]) ok = cudaMalloc(&buf[i], n[i]) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            for (uint8_t* b : buf)
                if (b) cudaFree(b);
            c->w1 = c->w1_sf = c->w2 = c->w2_sf = nullptr;
            c->weights_set = false;
            c->maps_weights = false;
            return MM_ERR_CUDA;
        }
        c->w1 = buf[0];
        c->w1_sf = buf[1];
        c->w2 = buf[2];
        c->w2_sf = buf[3];
    }
    c->weights_set = false;     // until the re-layout below has completed
    if (n_w2 != P * H * I / 2) CK(cudaMemset(c->w2, 0, n_w2));       // absent halves of a ragged last group
    CK(mm::launch_tile_weights(w1, c->w1, static_cast<int64_t>(P * 2 * I), c->H, o1, nullptr));
    CK(mm::launch_tile_weights(w2, c->w2, static_cast<int64_t>(P * H), c->I, o2, nullptr));
    CK(mm::launch_tile_scales(w1s, c->w1_sf, static_cast<int64_t>(P * 2 * I), c->H, o1, nullptr));
    CK(mm::launch_tile_scales(w2s, c->w2_sf, static_cast<int64_t>(P * H), c->I, o2, nullptr));
    CK(cudaDeviceSynchronize());
    if (!make_weight_map(&c->maps.w1, c->w1, b1, 2) || !make_weight_map(&c->maps.w2, c->w2, b2, 2) ||
        !make_weight_map(&c->maps.w2_one, c->w2, b2, 1) || !make_weight_map(&c->maps.w1_one, c->w1, b1, 1) ||
        !make_sf_map(&c->maps.w1_sf, c->w1_sf, b1, 4) || !make_sf_map(&c->maps.w2_sf, c->w2_sf, b2, 4))
        return MM_ERR_CUDA;
    c->maps_weights = true;
    c->weights_set = true;
    return MM_OK;
}

mm_status mm_set_eplb_map(mm_handle c, const int32_t* pol, const int32_t* rc, int R)
{
    if (!c || !pol || !rc || R < 1 || R > c->P) return MM_ERR_INVALID_ARG;
    std::vector<int> seen(c->P, 0);
    for (int e = 0; e < c->E; ++e) {
        if (rc[e] < 1 || rc[e] > R) return MM_ERR_INVALID_ARG;
        for (int s = 0; s < rc[e]; ++s) {
            const int p = pol[static_cast<int64_t>(e) * R + s];
            if (p < 0 || p >= c->P || seen[p]) return MM_ERR_INVALID_ARG;
            seen[p] = 1;
        }
    }
    for (int p = 0; p < c->P; ++p)
        if (!seen[p]) return MM_ERR_INVALID_ARG;
    if (capturing(nullptr)) return MM_ERR_INVALID_ARG;
    std::vector<int32_t> m(static_cast<size_t>(c->E) * R);
    for (int e = 0; e < c->E; ++e)
        for (int s = 0; s < R; ++s) m[static_cast<size_t>(e) * R + s] = s < rc[e] ? pol[e * R + s] : 0;
    int32_t *dm = nullptr, *drc = nullptr;
    if (cudaMalloc(&dm, m.size() * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&drc, c->E * sizeof(int32_t)) != cudaSuccess) {
        cudaGetLastError();
        if (dm) cudaFree(dm);
        return MM_ERR_CUDA;
    }
    if (cudaMemcpy(dm, m.data(), m.size() * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(drc, rc, c->E * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(dm);
        cudaFree(drc);
        return MM_ERR_CUDA;
    }
#ifdef MM_DEBUG
    if (c->fault == mm::kFaultMapEntry) {
        // the validated map's entry (logical 0, replica 0) overwritten on the
        // device with a physical id past the last expert
        const int32_t bad = c->P + 7;
        if (cudaMemcpy(dm, &bad, sizeof(bad), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(dm);
            cudaFree(drc);
            return MM_ERR_CUDA;
        }
    }
#endif
    cudaDeviceSynchronize();
    if (c->map) cudaFree(c->map);
    if (c->rc) cudaFree(c->rc);
    c->map = dm;
    c->rc = drc;
    c->R = R;
    c->host_map = m;
    c->host_rc.assign(rc, rc + c->E);
    c->map_set = true;
    return MM_OK;
}

mm_status mm_plan_replicas(const int64_t* load, int E, int P, int max_replicas, int32_t* pol, int32_t* rc)
{
    if (!load || !pol || !rc || E < 1 || P < E || P > MM_MAX_EXPERTS || max_replicas < 1) return MM_ERR_INVALID_ARG;
    if (P - E > static_cast<int64_t>(E) * (max_replicas - 1)) return MM_ERR_INVALID_ARG;
    for (int e = 0; e < E; ++e)
        if (load[e] < 0) return MM_ERR_INVALID_ARG;
    for (int64_t i = 0; i < static_cast<int64_t>(E) * max_replicas; ++i) pol[i] = -1;
    for (int e = 0; e < E; ++e) {
        pol[static_cast<int64_t>(e) * max_replicas] = e;       // every expert keeps its own slot
        rc[e] = 1;
    }
    for (int slot = E; slot < P; ++slot) {
        // the expert with the highest load per replica (exact: cross-multiplied), lower index on ties
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (rc[e] >= max_replicas) continue;
            if (best < 0) {
                best = e;
                continue;
            }
            const __int128 lhs = static_cast<__int128>(load[e]) * rc[best];
            const __int128 rhs = static_cast<__int128>(load[best]) * rc[e];
            if (lhs > rhs) best = e;
        }
        pol[static_cast<int64_t>(best) * max_replicas + rc[best]] = slot;
        rc[best] += 1;
    }
    return MM_OK;
}

mm_status mm_rebalance(mm_handle c, int layer, int max_replicas)
{
    if (!c || layer < 0 || layer >= MM_MAX_LAYERS || max_replicas < 1) return MM_ERR_INVALID_ARG;
    if (c->ep) return MM_ERR_UNSUPPORTED;
    if (!c->weights_set || !c->map_set) return MM_ERR_NOT_READY;
    if (c->P == c->E) return MM_OK;
    if (capturing(nullptr)) return MM_ERR_INVALID_ARG;
    std::vector<int64_t> load(c->E);
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(load.data(), c->counts + static_cast<int64_t>(layer) * c->E, sizeof(int64_t) * c->E,
                  cudaMemcpyDeviceToHost));
    std::vector<int32_t> pol(static_cast<size_t>(c->E) * max_replicas), rc(c->E);
    mm_status st = mm_plan_replicas(load.data(), c->E, c->P, max_replicas, pol.data(), rc.data());
    if (st != MM_OK) return st;
    // which logical expert each physical slot holds now, and will hold
    std::vector<int> now(c->P, -1), next(c->P, -1);
    for (int e = 0; e < c->E; ++e) {
        for (int r = 0; r < c->host_rc[e]; ++r) now[c->host_map[static_cast<size_t>(e) * c->R + r]] = e;
        for (int r = 0; r < rc[e]; ++r) next[pol[static_cast<size_t>(e) * max_replicas + r]] = e;
    }
    for (int e = 0; e < c->E; ++e)
        if (now[e] != e) return MM_ERR_NOT_READY;              // slot e must hold logical e (the copy source)
    // copy the weights of every slot whose logical expert changes from that expert's own slot
    const mm::WOrder o1 = mm::w1_order(c->H, c->I), o2 = mm::w2_order(c->H, c->I);
    const size_t e1 = mm::w_blocks(o1, 1), e2 = mm::w_blocks(o2, 1);   // blocks per expert
    for (int p = c->E; p < c->P; ++p) {
        if (now[p] == next[p]) continue;
        const int src = next[p];
        CK(cudaMemcpy(c->w1 + p * e1 * 8192, c->w1 + src * e1 * 8192, e1 * 8192, cudaMemcpyDeviceToDevice));
        CK(cudaMemcpy(c->w1_sf + p * e1 * 512, c->w1_sf + src * e1 * 512, e1 * 512, cudaMemcpyDeviceToDevice));
        CK(cudaMemcpy(c->w2 + p * e2 * 8192, c->w2 + src * e2 * 8192, e2 * 8192, cudaMemcpyDeviceToDevice));
        CK(cudaMemcpy(c->w2_sf + p * e2 * 512, c->w2_sf + src * e2 * 512, e2 * 512, cudaMemcpyDeviceToDevice));
    }
    CK(cudaDeviceSynchronize());
    return mm_set_eplb_map(c, pol.data(), rc.data(), max_replicas);
}

mm_status mm_bind_layer(mm_handle c, int layer)
{
    if (!c || layer < 0 || layer >= MM_MAX_LAYERS) return MM_ERR_INVALID_ARG;
    c->layer = layer;
    return MM_OK;
}

mm_status mm_set_recording(mm_handle c, int on)
{
    if (!c) return MM_ERR_INVALID_ARG;
    c->recording = on ? 1 : 0;
    return MM_OK;
}

mm_status mm_set_route(mm_handle c, mm_route r)
{
    if (!c || (r != MM_ROUTE_AUTO && r != MM_ROUTE_SMALL && r != MM_ROUTE_LARGE)) return MM_ERR_INVALID_ARG;
    c->route = r;
    return MM_OK;
}

mm_status mm_set_activation_format(mm_handle c, mm_act act)
{
    if (!c || (act != MM_ACT_MXFP8 && act != MM_ACT_BF16)) return MM_ERR_INVALID_ARG;
    if (act == c->act) return MM_OK;
    if (c->ep) return MM_ERR_UNSUPPORTED;
    if (capturing(nullptr)) return MM_ERR_INVALID_ARG;
    cudaDeviceSynchronize();
    free_ws(c);
    c->cap_tokens = 0;
    c->maps_ws = false;
    c->act = act;
    return MM_OK;
}

mm_status mm_set_shared_experts(mm_handle c, int num_shared)
{
    if (!c || num_shared < 0 || c->k + num_shared > MM_MAX_TOPK || c->P + num_shared > MM_MAX_EXPERTS)
        return MM_ERR_INVALID_ARG;
    if (num_shared == c->ns) return MM_OK;
    if (c->ep) return MM_ERR_UNSUPPORTED;
    if (capturing(nullptr)) return MM_ERR_INVALID_ARG;
    cudaDeviceSynchronize();
    // every per-expert and per-pair size changes: weights and workspace go
    free_ws(c);
    c->cap_tokens = 0;
    c->maps_ws = false;
    cudaFree(c->w1);
    cudaFree(c->w1_sf);
    cudaFree(c->w2);
    cudaFree(c->w2_sf);
    c->w1 = c->w2 = c->w1_sf = c->w2_sf = nullptr;
    c->weights_set = false;
    c->maps_weights = false;
    c->ns = num_shared;
    return MM_OK;
}

mm_status mm_reserve(mm_handle c, int64_t max_tokens)
{
    if (!c || max_tokens < 0 || max_tokens > (int64_t(1) << 24)) return MM_ERR_INVALID_ARG;
    if (max_tokens <= c->cap_tokens) return MM_OK;
    if (capturing(nullptr)) return MM_ERR_INVALID_ARG;
    return mm::reserve_pairs(c, max_tokens * mm::slots(c), max_tokens);
}

}  // extern "C"

// The workspace for up to `npairs` (token, slot) pairs -- or received rows
// under expert parallelism -- over the routing's physical experts, and for
// forwards of up to `max_tokens` tokens.
mm_status mm::reserve_pairs(mm_handle c, int64_t npairs, int64_t max_tokens)
{
    const int kk = mm::slots(c), P = mm::pw(c);              // slots per token, physical experts
    // each non-empty segment adds < kSegAlign pad rows and < 1 partial token tile
    const int64_t busy = npairs < P ? npairs : P;
    const int64_t rows = npairs + busy * (mm::kSegAlign - 1) + mm::kSegAlign;
    // token tiles: kTokTile rows on the large-input path, kSmallTile rows in the fused kernel
    const int64_t small_pairs = npairs < int64_t(mm::kSmallMaxTokens) * kk ? npairs : int64_t(mm::kSmallMaxTokens) * kk;
    const int64_t tiles = std::max(npairs / mm::kTokTile, small_pairs / mm::kSmallTile) + busy + 1;
    const int64_t chunks = (npairs + mm::kChunkPairs - 1) / mm::kChunkPairs;
    const int64_t H = c->H, I = c->I;
    // size pass, then carve
    size_t bytes = 0;
    auto add = [&](size_t n) { bytes += (n + 255) & ~size_t(255); };
    add(npairs * 4 * 4);                      // idx, phys, pos, wgt
    add(chunks * P * 4);
    add((P + 1) * 4);
    add(P * 4);                               // first tile of each expert
    add(tiles * 4 * 4 + 16);                  // tile table, done1, num_tiles, unit counter, pair count
    add(tiles * 2 * 4);                       // tile pairs
    const int64_t eb = c->act == MM_ACT_BF16 ? 2 : 1;     // bytes per dispatched activation element
    add(rows * H * eb);
    add(tiles * (H / 128) * 512);
    add(rows * I * eb);
    add(tiles * (I / 128) * 512);
    add(rows * H * 2);
    add(64);                                  // grid barrier
    add(static_cast<size_t>(c->sms) * 8 * 8); // stage timestamps
    bytes += 8 * 256;
    cudaDeviceSynchronize();
    free_ws(c);
    void* ws = nullptr;
    if (cudaMalloc(&ws, bytes) != cudaSuccess) {
        cudaGetLastError();
        return MM_ERR_CUDA;
    }
    CK(cudaMemset(ws, 0, bytes));
    uint8_t* p = static_cast<uint8_t*>(ws);
    c->idx = carve<int32_t>(p, npairs);
    c->phys = carve<int32_t>(p, npairs);
    c->pos = carve<int32_t>(p, npairs);
    c->wgt = carve<float>(p, npairs);
    c->chunk_hist = carve<int32_t>(p, chunks * P);
    c->off = carve<int32_t>(p, P + 1);
    c->toff = carve<int32_t>(p, P);
    c->tile_expert = carve<int32_t>(p, tiles);
    c->tile_row0 = carve<int32_t>(p, tiles);
    c->tile_rows = carve<int32_t>(p, tiles);
    c->done1 = carve<int32_t>(p, tiles);
    c->num_tiles = carve<int32_t>(p, 4);
    c->unit_next = c->num_tiles + 1;
    c->st_tile = carve<int32_t>(p, tiles * 2);
    c->xq = carve<uint8_t>(p, rows * H * eb);
    c->xs_t = carve<uint8_t>(p, tiles * (H / 128) * 512);
    c->hq = carve<uint8_t>(p, rows * I * eb);
    c->hs_t = carve<uint8_t>(p, tiles * (I / 128) * 512);
    c->y = carve<__nv_bfloat16>(p, rows * H);
    c->grid_bar = carve<unsigned>(p, 16);
    c->stamps = carve<uint64_t>(p, static_cast<size_t>(c->sms) * 8);
    c->ws = ws;
    c->ws_bytes = bytes;
    for (int i = 0; i < mm::kTokBoxes; ++i) {
        bool ok;
        if (c->act == MM_ACT_BF16)
            ok = make_map(&c->maps16.xd[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c->xq, H, rows, H * 2, mm::kBBox << i,
                          64) &&
                 make_map(&c->maps16.hb[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c->hq, I, rows, I * 2, mm::kBBox << i,
                          64);
        else
            ok = make_sf_map(&c->maps.xs_sf, c->xs_t, tiles * (H / 128), 2) &&
                 make_sf_map(&c->maps.hs_sf, c->hs_t, tiles * (I / 128), 2) &&
                 make_map(&c->maps.xq[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, c->xq, H, rows, H, mm::kBBox << i) &&
                 make_map(&c->maps.hq[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, c->hq, I, rows, I, mm::kBBox << i);
        if (!ok) {
            free_ws(c);
            return MM_ERR_CUDA;
        }
    }
    c->ws_act = c->act;
    c->cap_tokens = max_tokens;
    c->rows_cap = rows;
    c->tiles_cap = tiles;
    c->chunks_cap = chunks;
    c->maps_ws = true;
    return MM_OK;
}

extern "C" {

mm_status mm_forward(mm_handle c, const void* hidden, const float* logits, const float* bias, void* out,
                     int64_t T, mm_stream stream)
{
    if (!c || T < 0) return MM_ERR_INVALID_ARG;
    if (c->ep) return MM_ERR_UNSUPPORTED;       // an expert-parallel rank runs mm_ep_dispatch / _experts / _combine
    if (!c->weights_set || !c->map_set) return MM_ERR_NOT_READY;
    if (T == 0) return MM_OK;
    if (!hidden || !logits || !out) return MM_ERR_INVALID_ARG;
    if (!aligned(hidden, 16) || !aligned(out, 16) || !aligned(logits, 4) || (bias && !aligned(bias, 4)))
        return MM_ERR_INVALID_ARG;
    if (T > c->cap_tokens) return MM_ERR_CAPACITY;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool prof16 = c->prof_used < static_cast<int>(c->prof_events.size()) / 2;
    if (c->act == MM_ACT_BF16) {
        // a16w4: the multi-launch path with bf16 dispatch and the bf16 x MXFP4 GEMM
        if (c->route == MM_ROUTE_SMALL) return MM_ERR_UNSUPPORTED;
        if (mm::launch_route(c, logits, bias, T, s) != cudaSuccess) return MM_ERR_CUDA;
        if (mm::launch_permute(c, T, s) != cudaSuccess) return MM_ERR_CUDA;
        if (mm::launch_dispatch16(c, hidden, T, s) != cudaSuccess) return MM_ERR_CUDA;
        if (prof16 && cudaEventRecord(c->prof_events[2 * c->prof_used], s) != cudaSuccess) return MM_ERR_CUDA;
        if (mm::launch_gemm16(c, s) != cudaSuccess) return MM_ERR_CUDA;
        if (prof16 && cudaEventRecord(c->prof_events[2 * c->prof_used + 1], s) != cudaSuccess) return MM_ERR_CUDA;
        if (mm::launch_combine(c, out, T, s) != cudaSuccess) return MM_ERR_CUDA;
        if (prof16) ++c->prof_used;
        c->last_route = 2;
        c->last_launches = 7;
        c->last_gemm = 3;
        c->last_T = T;
        c->last_stream = s;
        return MM_OK;
    }
    if (c->route == MM_ROUTE_SMALL && T > c->small_max) return MM_ERR_CAPACITY;
    const bool small = c->route == MM_ROUTE_SMALL || (c->route == MM_ROUTE_AUTO && T <= c->small_max);
    const bool prof = c->prof_used < static_cast<int>(c->prof_events.size()) / 2;
    if (small) {
        // one cooperative launch: every stage of the layer
        if (prof && cudaEventRecord(c->prof_events[2 * c->prof_used], s) != cudaSuccess) return MM_ERR_CUDA;
        if (mm::launch_small(c, hidden, logits, bias, out, T, s) != cudaSuccess) return MM_ERR_CUDA;
        if (prof && cudaEventRecord(c->prof_events[2 * c->prof_used + 1], s) != cudaSuccess) return MM_ERR_CUDA;
    } else {
        if (mm::launch_route(c, logits, bias, T, s) != cudaSuccess) return MM_ERR_CUDA;
        if (mm::launch_permute(c, T, s) != cudaSuccess) return MM_ERR_CUDA;
        if (mm::launch_quant_dispatch(c, hidden, T, s) != cudaSuccess) return MM_ERR_CUDA;
        if (prof && cudaEventRecord(c->prof_events[2 * c->prof_used], s) != cudaSuccess) return MM_ERR_CUDA;
        if (mm::launch_gemm(c, T, s) != cudaSuccess) return MM_ERR_CUDA;
        if (prof && cudaEventRecord(c->prof_events[2 * c->prof_used + 1], s) != cudaSuccess) return MM_ERR_CUDA;
        if (mm::launch_combine(c, out, T, s) != cudaSuccess) return MM_ERR_CUDA;
    }
    if (prof) ++c->prof_used;
    c->last_route = small ? 1 : 2;
    c->last_gemm = small ? 0 : mm::gemm_kind(c);
    c->last_launches = small ? 1 : (c->last_gemm == 4 ? 8 : 7);
    c->last_T = T;
    c->last_stream = s;
    return MM_OK;
}

mm_status mm_profile_begin(mm_handle c, int max_launches)
{
    if (!c || max_launches < 1 || max_launches > 100000) return MM_ERR_INVALID_ARG;
    profile_free(c);
    c->prof_events.resize(2 * static_cast<size_t>(max_launches));
    for (auto& e : c->prof_events) {
        if (cudaEventCreate(&e) != cudaSuccess) {
            cudaGetLastError();
            e = nullptr;
            profile_free(c);
            return MM_ERR_CUDA;
        }
    }
    return MM_OK;
}

mm_status mm_profile_end(mm_handle c, float* ms_out, int max_out, int* n_out)
{
    if (!c || !n_out || (max_out > 0 && !ms_out)) return MM_ERR_INVALID_ARG;
    *n_out = 0;
    CK(cudaDeviceSynchronize());
    const int n = c->prof_used < max_out ? c->prof_used : max_out;
    for (int i = 0; i < n; ++i) CK(cudaEventElapsedTime(&ms_out[i], c->prof_events[2 * i], c->prof_events[2 * i + 1]));
    *n_out = n;
    profile_free(c);
    return MM_OK;
}

mm_status mm_read_counts(mm_handle c, int layer, int64_t* out_host)
{
    if (!c || !out_host || layer < 0 || layer >= MM_MAX_LAYERS) return MM_ERR_INVALID_ARG;
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(out_host, c->counts + static_cast<int64_t>(layer) * c->E, sizeof(int64_t) * c->E,
                  cudaMemcpyDeviceToHost));
    int code = 0;
    CK(cudaMemcpy(&code, c->status, sizeof(int), cudaMemcpyDeviceToHost));
    return static_cast<mm_status>(code);
}

mm_status mm_reset_counts(mm_handle c, int layer)
{
    if (!c || layer < -1 || layer >= MM_MAX_LAYERS) return MM_ERR_INVALID_ARG;
    CK(cudaDeviceSynchronize());
    if (layer < 0) CK(cudaMemset(c->counts, 0, sizeof(int64_t) * MM_MAX_LAYERS * c->E));
    else CK(cudaMemset(c->counts + static_cast<int64_t>(layer) * c->E, 0, sizeof(int64_t) * c->E));
    return MM_OK;
}

mm_status mm_get_status(mm_handle c, int* device_code)
{
    if (!c || !device_code) return MM_ERR_INVALID_ARG;
    CK(cudaDeviceSynchronize());
    int st[2] = {0, 0};
    CK(cudaMemcpy(st, c->status, sizeof(st), cudaMemcpyDeviceToHost));
    *device_code = st[0];
    c->last_site = st[1];
    CK(cudaMemset(c->status, 0, sizeof(st)));
    if (st[0] != 0 && c->grid_bar) CK(cudaMemset(c->grid_bar, 0, 16 * sizeof(unsigned)));
    return MM_OK;
}

static mm_status debug_geometry(mm_handle c, int stage, size_t* bytes, int32_t* rows_out)
{
    if (!c->ws || c->last_T == 0) {
        *bytes = 0;
        return MM_OK;
    }
    int32_t rows = 0;
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(&rows, c->off + mm::pw(c), sizeof(int32_t), cudaMemcpyDeviceToHost));
    *rows_out = rows;
    const size_t pairs = static_cast<size_t>(c->last_T) * mm::slots(c);
    const bool a16 = c->ws_act == MM_ACT_BF16;
    switch (stage) {
        case 0: case 1: case 2: case 3: *bytes = pairs * 4; break;
        case 4: *bytes = (mm::pw(c) + 1) * 4; break;
        case 5: *bytes = static_cast<size_t>(rows) * c->H * (a16 ? 2 : 1); break;
        case 6: *bytes = a16 ? 0 : static_cast<size_t>(rows) * c->H / 32; break;
        case 7: *bytes = static_cast<size_t>(rows) * c->I * (a16 ? 2 : 1); break;
        case 8: *bytes = a16 ? 0 : static_cast<size_t>(rows) * c->I / 32; break;
        case 9: *bytes = static_cast<size_t>(rows) * c->H * 2; break;
        case 10: *bytes = 4 * sizeof(int32_t); break;
        case 11: *bytes = static_cast<size_t>(c->sms) * 8 * sizeof(uint64_t); break;
        case 12: {
            int32_t ntiles = 0;
            CK(cudaMemcpy(&ntiles, c->num_tiles, sizeof(int32_t), cudaMemcpyDeviceToHost));
            *bytes = static_cast<size_t>(ntiles) * 3 * sizeof(int32_t);
            break;
        }
        default: return MM_ERR_INVALID_ARG;
    }
    return MM_OK;
}

mm_status mm_debug_size(mm_handle c, int stage, size_t* bytes)
{
    if (!c || !bytes) return MM_ERR_INVALID_ARG;
    int32_t rows = 0;
    return debug_geometry(c, stage, bytes, &rows);
}

mm_status mm_debug_dump(mm_handle c, int stage, void* dst, size_t bytes)
{
    if (!c || !dst) return MM_ERR_INVALID_ARG;
    size_t full = 0;
    int32_t rows = 0;
    mm_status st = debug_geometry(c, stage, &full, &rows);
    if (st != MM_OK) return st;
    const size_t n = bytes < full ? bytes : full;
    if (n == 0) return MM_OK;
    if (stage == 10) {
        int32_t site = 0;
        CK(cudaMemcpy(&site, c->status + 1, sizeof(int32_t), cudaMemcpyDeviceToHost));
        int32_t kind = c->last_gemm;
        if (kind == 4) {
            // both large-input GEMM kernels were launched; the tile scan chose one
            int32_t pairs = 0;
            CK(cudaMemcpy(&pairs, c->num_tiles + 3, sizeof(int32_t), cudaMemcpyDeviceToHost));
            kind = pairs ? 2 : 1;
        }
        const int32_t info[4] = {c->last_route, c->last_launches, site ? site : c->last_site, kind};
        memcpy(dst, info, n);
        return MM_OK;
    }
    if (stage == 12) {
        const size_t ntiles = full / (3 * sizeof(int32_t));
        std::vector<int32_t> cols(3 * ntiles), table(3 * ntiles);
        CK(cudaMemcpy(cols.data(), c->tile_expert, ntiles * sizeof(int32_t), cudaMemcpyDeviceToHost));
        CK(cudaMemcpy(cols.data() + ntiles, c->tile_row0, ntiles * sizeof(int32_t), cudaMemcpyDeviceToHost));
        CK(cudaMemcpy(cols.data() + 2 * ntiles, c->tile_rows, ntiles * sizeof(int32_t), cudaMemcpyDeviceToHost));
        for (size_t t = 0; t < ntiles; ++t)
            for (int j = 0; j < 3; ++j) table[3 * t + j] = cols[j * ntiles + t];
        memcpy(dst, table.data(), n);
        return MM_OK;
    }
    const void* src = nullptr;
    switch (stage) {
        case 0: src = c->idx; break;
        case 1: src = c->wgt; break;
        case 2: src = c->phys; break;
        case 3: src = c->pos; break;
        case 4: src = c->off; break;
        case 5: src = c->xq; break;
        case 7: src = c->hq; break;
        case 9: src = c->y; break;
        case 11: src = c->stamps; break;
        default: break;
    }
    if (src) {
        CK(cudaMemcpy(dst, src, n, cudaMemcpyDeviceToHost));
        return MM_OK;
    }
    // scale stages: per-token-tile scale tiles -> row-major [rows][K/32] (pad rows 0)
    const int K = stage == 6 ? c->H : c->I;
    const int nb = K / 32;
    const uint8_t* tiled = stage == 6 ? c->xs_t : c->hs_t;
    int32_t ntiles = 0;
    CK(cudaMemcpy(&ntiles, c->num_tiles, sizeof(int32_t), cudaMemcpyDeviceToHost));
    std::vector<int32_t> row0(ntiles), trows(ntiles);
    std::vector<uint8_t> t(static_cast<size_t>(ntiles) * (K / 128) * 512);
    if (ntiles > 0) {
        CK(cudaMemcpy(row0.data(), c->tile_row0, ntiles * sizeof(int32_t), cudaMemcpyDeviceToHost));
        CK(cudaMemcpy(trows.data(), c->tile_rows, ntiles * sizeof(int32_t), cudaMemcpyDeviceToHost));
        CK(cudaMemcpy(t.data(), tiled, t.size(), cudaMemcpyDeviceToHost));
    }
    uint8_t* d = static_cast<uint8_t*>(dst);
    memset(d, 0, n);
    for (int32_t tile = 0; tile < ntiles; ++tile)
        for (int r = 0; r < trows[tile]; ++r)
            for (int b = 0; b < nb; ++b) {
                const size_t at = static_cast<size_t>(row0[tile] + r) * nb + b;
                if (at < n) d[at] = t[mm::act_sf_offset(tile, r, b, K / 128)];
            }
    return MM_OK;
}

}  // extern "C"
