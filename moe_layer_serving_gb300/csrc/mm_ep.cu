// mm_ep.cu -- the layer forward under expert parallelism: the physical
// experts are split over ranks, and the dispatch and the combine become an
// exchange of rows between them (the pages run the fused operator expert-
// parallel over eight GPUs, with all-to-all dispatch and combine buffers,
// "sglang PR #35619", launch settings; "sglang PR #47065", Title/switches).
//
// One rank's forward is four steps, of which the library runs three; the
// exchanges between them are the caller's (NCCL all-to-all, or copies):
//
//   mm_ep_dispatch   route + EPLB remap + record, permute by physical expert,
//                    MXFP8-quantise each token into its k rows of the send
//                    buffer; rows for rank d form one contiguous range, the
//                    segments of d's experts in expert order
//   (exchange)       rank d receives its ranges from every source rank
//   mm_ep_experts    permute the received rows by the rank's own experts, the
//                    grouped GEMM1 (+SwiGLU, requant) and GEMM2 over them, and
//                    gather y back into the order the rows were received
//   (exchange)       each y row returns to the rank that sent its token
//   mm_ep_combine    out[t] = bf16(sum_j w[t,j] y[row of (t,j)]) in slot order
//
// The arithmetic of every row is the single-GPU forward's: the same codes,
// scales, MMAs and epilogue, and the same combine order, so a layer run
// expert-parallel gives the single-GPU output bit for bit.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <vector>

#include "mm_device.cuh"
#include "mm_internal.h"
#include "mm_stages.cuh"

namespace mm {
namespace {

// Quantise block b of token t once and write it into the token's k rows of
// the send buffer: codes [row][H], scales row-major [row][H/32], and (block 0)
// the destination's local expert index of the row.
__global__ void __launch_bounds__(256) ep_pack_kernel(const __nv_bfloat16* __restrict__ x, int64_t T, int H, int k,
                                                      const int32_t* __restrict__ pos,
                                                      const int32_t* __restrict__ phys,
                                                      const int32_t* __restrict__ local_id,
                                                      uint8_t* __restrict__ send_xq, uint8_t* __restrict__ send_xs,
                                                      int32_t* __restrict__ send_eid, DispatchBounds chk)
{
    const int nb = H / 32;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t t = g / nb;
    if (t >= T) return;
    const int b = static_cast<int>(g % nb);
    uint32_t packed[8];
    const uint8_t sbyte = quant_block32(x, t, b, H, packed);
    for (int j = 0; j < k; ++j) {
        const int64_t row = pos[t * k + j];
        const int p = phys[t * k + j];
        if (!MM_CHECK(p >= 0 && p < chk.P && row >= 0 && row < chk.rows_cap, chk.status, kSiteDispatch)) continue;
        uint4* dst = reinterpret_cast<uint4*>(send_xq + row * H + b * 32);
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        send_xs[row * nb + b] = sbyte;
        if (b == 0) send_eid[row] = local_id[p];
    }
}

// Received row i (local expert e = eid[i], -1 = a padding row) moves to its
// dispatch row rpos[i]: 32 codes per thread, and the scale byte into the
// scale tile of the row's token tile.
__global__ void __launch_bounds__(256) ep_unpack_kernel(const uint8_t* __restrict__ recv_xq,
                                                        const uint8_t* __restrict__ recv_xs,
                                                        const int32_t* __restrict__ eid, int64_t n, int H,
                                                        const int32_t* __restrict__ rpos,
                                                        const int32_t* __restrict__ off,
                                                        const int32_t* __restrict__ toff, uint8_t* __restrict__ xq,
                                                        uint8_t* __restrict__ xs_t, DispatchBounds chk)
{
    const int nb = H / 32;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t i = g / nb;
    if (i >= n) return;
    const int b = static_cast<int>(g % nb);
    const int e = eid[i];
    if (e < 0) return;
    const int64_t row = rpos[i];
    if (!MM_CHECK(e < chk.P && row >= 0 && row < chk.rows_cap, chk.status, kSiteDispatch)) return;
    const uint4* src = reinterpret_cast<const uint4*>(recv_xq + i * H + b * 32);
    uint4* dst = reinterpret_cast<uint4*>(xq + row * H + b * 32);
    const uint4 a0 = src[0], a1 = src[1];
    dst[0] = a0;
    dst[1] = a1;
    const int rank = static_cast<int>(row) - off[e];
    xs_t[act_sf_offset(toff[e] + rank / kTokTile, rank % kTokTile, b, H / 128)] = recv_xs[i * nb + b];
}

// y of received row i, in the order the rows were received (zeros for a
// padding row): 16 bytes per thread.
__global__ void __launch_bounds__(256) ep_gather_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ eid,
                                                        const int32_t* __restrict__ rpos, int64_t n, int H,
                                                        uint4* __restrict__ y_recv, DispatchBounds chk)
{
    const int nc = H / 8;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t i = g / nc;
    if (i >= n) return;
    const int c = static_cast<int>(g % nc);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (eid[i] >= 0) {
        const int64_t row = rpos[i];
        if (MM_CHECK(row >= 0 && row < chk.rows_cap, chk.status, kSiteCombine)) v = y[row * nc + c];
    }
    y_recv[i * nc + c] = v;
}

__global__ void __launch_bounds__(256) ep_combine_kernel(const __nv_bfloat16* __restrict__ y,
                                                         const float* __restrict__ w,
                                                         const int32_t* __restrict__ pos, int64_t T, int H, int k,
                                                         __nv_bfloat16* __restrict__ out, DispatchBounds chk)
{
    const int nc = H / 8;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t t = g / nc;
    if (t >= T) return;
    combine_chunk(y, w, pos, t, static_cast<int>(g % nc), H, k, out, chk);
}

unsigned blocks_for(int64_t threads) { return static_cast<unsigned>((threads + 255) / 256); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// rows of the send buffer for T tokens: T k pairs plus each segment's padding
int64_t send_rows(const mm_ctx* c, int64_t T)
{
    const int64_t npairs = T * c->k;
    const int64_t busy = npairs < c->P ? npairs : c->P;
    return npairs + busy * (kSegAlign - 1) + kSegAlign;
}

bool on_capture(cudaStream_t s)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return st != cudaStreamCaptureStatusNone;
}

void ep_free(mm_ctx* c)
{
    if (c->ep_recv_pos) cudaFree(c->ep_recv_pos);
    c->ep_recv_pos = nullptr;
    c->ep_recv_cap = 0;
}

}  // namespace

void ep_release(mm_ctx* c)
{
    ep_free(c);
    if (c->ep_local_id) cudaFree(c->ep_local_id);
    c->ep_local_id = nullptr;
}

}  // namespace mm

extern "C" {

mm_status mm_set_expert_parallel(mm_handle c, int rank, int world, const int32_t* first)
{
    if (!c || world < 1 || world > MM_MAX_EXPERTS || rank < 0 || rank >= world || !first) return MM_ERR_INVALID_ARG;
    if (first[0] != 0 || first[world] != c->P) return MM_ERR_INVALID_ARG;
    for (int r = 0; r < world; ++r)
        if (first[r + 1] <= first[r]) return MM_ERR_INVALID_ARG;      // every rank owns at least one expert
    if (c->ns != 0 || c->act != MM_ACT_MXFP8) return MM_ERR_UNSUPPORTED;
    if (mm::on_capture(nullptr)) return MM_ERR_INVALID_ARG;
    std::vector<int32_t> local(c->P);
    for (int r = 0; r < world; ++r)
        for (int p = first[r]; p < first[r + 1]; ++p) local[p] = p - first[r];
    int32_t* d = nullptr;
    if (cudaMalloc(&d, sizeof(int32_t) * c->P) != cudaSuccess ||
        cudaMemcpy(d, local.data(), sizeof(int32_t) * c->P, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        if (d) cudaFree(d);
        return MM_ERR_CUDA;
    }
    cudaDeviceSynchronize();
    // the weights and the workspace were sized for the whole expert set
    mm::ep_release(c);
    void* w[] = {c->w1, c->w1_sf, c->w2, c->w2_sf};
    for (void* p : w)
        if (p) cudaFree(p);
    c->w1 = c->w1_sf = c->w2 = c->w2_sf = nullptr;
    c->weights_set = false;
    c->maps_weights = false;
    if (c->ws) {
        cudaFree(c->ws);
        c->ws = nullptr;
        c->ws_bytes = 0;
    }
    c->cap_tokens = 0;
    c->maps_ws = false;
    c->ep = true;
    c->ep_rank = rank;
    c->ep_world = world;
    c->ep_local = first[rank + 1] - first[rank];
    c->ep_first.assign(first, first + world + 1);
    c->ep_local_id = d;
    return MM_OK;
}

mm_status mm_ep_reserve(mm_handle c, int64_t max_tokens, int64_t max_recv_rows)
{
    if (!c || !c->ep || max_tokens < 0 || max_tokens > (int64_t(1) << 24) || max_recv_rows < 0 ||
        max_recv_rows > (int64_t(1) << 27))
        return MM_ERR_INVALID_ARG;
    if (max_tokens <= c->cap_tokens && max_recv_rows <= c->ep_recv_cap) return MM_OK;
    if (mm::on_capture(nullptr)) return MM_ERR_INVALID_ARG;
    cudaDeviceSynchronize();
    mm::ep_free(c);
    const int64_t tokens = max_tokens > c->cap_tokens ? max_tokens : c->cap_tokens;
    const int64_t pairs = tokens * c->k > max_recv_rows ? tokens * c->k : max_recv_rows;
    mm_status st = mm::reserve_pairs(c, pairs, tokens);
    if (st != MM_OK) return st;
    if (max_recv_rows > 0 && cudaMalloc(&c->ep_recv_pos, sizeof(int32_t) * max_recv_rows) != cudaSuccess) {
        cudaGetLastError();
        c->ep_recv_pos = nullptr;
        return MM_ERR_CUDA;
    }
    c->ep_recv_cap = max_recv_rows;
    return MM_OK;
}

mm_status mm_ep_send_rows(mm_handle c, int64_t num_tokens, int64_t* rows)
{
    if (!c || !c->ep || num_tokens < 0 || !rows) return MM_ERR_INVALID_ARG;
    *rows = num_tokens == 0 ? 0 : mm::send_rows(c, num_tokens);
    return MM_OK;
}

mm_status mm_ep_dispatch(mm_handle c, const void* hidden, const float* logits, const float* bias, int64_t T,
                         void* send_xq, void* send_xs, int32_t* send_eid, int64_t send_capacity, int64_t* row_off,
                         mm_stream stream)
{
    if (!c || T < 0 || !row_off || send_capacity < 0) return MM_ERR_INVALID_ARG;
    if (!c->ep) return MM_ERR_NOT_READY;
    if (!c->map_set) return MM_ERR_NOT_READY;
    if (T > c->cap_tokens) return MM_ERR_CAPACITY;
    if (T == 0) {
        for (int d = 0; d <= c->ep_world; ++d) row_off[d] = 0;
        c->ep_T = 0;
        c->ep_send_rows = 0;
        return MM_OK;
    }
    if (!hidden || !logits || !send_xq || !send_xs || !send_eid) return MM_ERR_INVALID_ARG;
    if (!mm::aligned16(hidden) || !mm::aligned16(send_xq) || (reinterpret_cast<uintptr_t>(logits) & 3) ||
        (bias && (reinterpret_cast<uintptr_t>(bias) & 3)) || (reinterpret_cast<uintptr_t>(send_eid) & 3))
        return MM_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (mm::on_capture(s)) return MM_ERR_INVALID_ARG;          // reads the split sizes back to the host
    const int64_t rows = mm::send_rows(c, T);
    if (rows > send_capacity) return MM_ERR_CAPACITY;
    if (cudaMemsetAsync(send_eid, 0xFF, sizeof(int32_t) * rows, s) != cudaSuccess) return MM_ERR_CUDA;
    if (mm::launch_route(c, logits, bias, T, s) != cudaSuccess) return MM_ERR_CUDA;
    if (mm::launch_permute(c, T, s) != cudaSuccess) return MM_ERR_CUDA;
    const mm::DispatchBounds chk{c->P, rows, c->status};
    mm::ep_pack_kernel<<<mm::blocks_for(T * (c->H / 32)), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(hidden), T, c->H, c->k, c->pos, c->phys, c->ep_local_id,
        static_cast<uint8_t*>(send_xq), static_cast<uint8_t*>(send_xs), send_eid, chk);
    if (cudaGetLastError() != cudaSuccess) return MM_ERR_CUDA;
    std::vector<int32_t> off(c->P + 1);
    if (cudaMemcpyAsync(off.data(), c->off, sizeof(int32_t) * (c->P + 1), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return MM_ERR_CUDA;
    }
    for (int d = 0; d <= c->ep_world; ++d) row_off[d] = off[c->ep_first[d]];
    c->ep_T = T;
    c->ep_send_rows = rows;
    c->last_T = T;
    c->last_route = 2;
    c->last_stream = s;
    return MM_OK;
}

mm_status mm_ep_experts(mm_handle c, const void* recv_xq, const void* recv_xs, const int32_t* recv_eid, int64_t n,
                        void* y_recv, mm_stream stream)
{
    if (!c || n < 0) return MM_ERR_INVALID_ARG;
    if (!c->ep || !c->weights_set) return MM_ERR_NOT_READY;
    if (n > c->ep_recv_cap) return MM_ERR_CAPACITY;
    if (n == 0) return MM_OK;
    if (!recv_xq || !recv_xs || !recv_eid || !y_recv || !mm::aligned16(recv_xq) || !mm::aligned16(y_recv) ||
        (reinterpret_cast<uintptr_t>(recv_eid) & 3))
        return MM_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const mm::DispatchBounds chk{c->ep_local, c->rows_cap, c->status};
    if (mm::launch_permute_ids(c, recv_eid, n, c->ep_local, c->ep_recv_pos, s) != cudaSuccess) return MM_ERR_CUDA;
    mm::ep_unpack_kernel<<<mm::blocks_for(n * (c->H / 32)), 256, 0, s>>>(
        static_cast<const uint8_t*>(recv_xq), static_cast<const uint8_t*>(recv_xs), recv_eid, n, c->H,
        c->ep_recv_pos, c->off, c->toff, c->xq, c->xs_t, chk);
    if (cudaGetLastError() != cudaSuccess) return MM_ERR_CUDA;
    const bool prof = c->prof_used < static_cast<int>(c->prof_events.size()) / 2;
    if (prof && cudaEventRecord(c->prof_events[2 * c->prof_used], s) != cudaSuccess) return MM_ERR_CUDA;
    if (mm::launch_gemm(c, n, s) != cudaSuccess) return MM_ERR_CUDA;
    if (prof && cudaEventRecord(c->prof_events[2 * c->prof_used + 1], s) != cudaSuccess) return MM_ERR_CUDA;
    if (prof) ++c->prof_used;
    mm::ep_gather_kernel<<<mm::blocks_for(n * (c->H / 8)), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(c->y), recv_eid, c->ep_recv_pos, n, c->H, static_cast<uint4*>(y_recv), chk);
    if (cudaGetLastError() != cudaSuccess) return MM_ERR_CUDA;
    return MM_OK;
}

mm_status mm_ep_combine(mm_handle c, const void* y_back, void* out, mm_stream stream)
{
    if (!c) return MM_ERR_INVALID_ARG;
    if (!c->ep) return MM_ERR_NOT_READY;
    if (c->ep_T == 0) return MM_OK;
    if (!y_back || !out || !mm::aligned16(y_back) || !mm::aligned16(out)) return MM_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const mm::DispatchBounds chk{c->P, c->ep_send_rows, c->status};
    mm::ep_combine_kernel<<<mm::blocks_for(c->ep_T * (c->H / 8)), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(y_back), c->wgt, c->pos, c->ep_T, c->H, c->k,
        static_cast<__nv_bfloat16*>(out), chk);
    return cudaGetLastError() == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}

}  // extern "C"
