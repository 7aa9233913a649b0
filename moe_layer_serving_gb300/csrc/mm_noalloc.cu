// mm_noalloc.cu -- a dispatch planner that allocates nothing.
//
// Some callers cannot allocate device memory at the point where they need the
// dispatch plan: code that runs inside another framework's memory pool or
// allocator-free runtime, or a serving loop that must not call cudaMalloc
// (which synchronises the device) in its steady state.  For them this file
// provides one entry point whose scratch memory is a fixed array compiled into
// the library instead of caller- or library-allocated workspace.
//
// It is a single-CTA variant of the permute kernels (chunk histograms ->
// per-expert scan into aligned segments -> stable scatter), producing
// the same dispatch rows and segment offsets as mm_forward's permute.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mm_internal.h"

namespace {

constexpr int kPlanMaxPairs = 131072;                    // e.g. 16384 tokens x top-8
constexpr int kPlanChunk = 1024;                         // pairs per chunk histogram
constexpr int kPlanMaxChunks = kPlanMaxPairs / kPlanChunk;
constexpr int kPlanThreads = 1024;

// Per-chunk, per-expert counts (then running row bases): 128 x 512 x 4 B =
// 256 KB.  Every GPU that loads the library holds this array until the process
// exits.  All calls share it; each call overwrites the part it uses.
static __device__ __align__(256) int32_t g_plan_scratch[kPlanMaxChunks * MM_MAX_EXPERTS];

__global__ void __launch_bounds__(kPlanThreads, 1)
    plan_kernel(const int32_t* __restrict__ phys, int npairs, int P, int32_t* scratch, int32_t* __restrict__ pos,
                int32_t* __restrict__ off)
{
    __shared__ int cnt[MM_MAX_EXPERTS];
    __shared__ int soff[MM_MAX_EXPERTS + 1];
    const int nchunks = (npairs + kPlanChunk - 1) / kPlanChunk;
    // 1. clear the part of the shared scratch this call uses
    for (int i = threadIdx.x; i < nchunks * P; i += blockDim.x) scratch[i] = 0;
    __syncthreads();
    // 2. chunk histograms
    for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
        const int p = phys[i];
        if (p >= 0 && p < P) atomicAdd(&scratch[(i / kPlanChunk) * P + p], 1);
    }
    __syncthreads();
    // 3. per expert: exclusive bases over chunks, totals
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        int run = 0;
        for (int c = 0; c < nchunks; ++c) {
            const int v = scratch[c * P + p];
            scratch[c * P + p] = run;
            run += v;
        }
        cnt[p] = run;
    }
    __syncthreads();
    // 4. segment starts, each segment padded to the forward's segment alignment
    if (threadIdx.x == 0) {
        int o = 0;
        for (int p = 0; p < P; ++p) {
            soff[p] = o;
            o += mm::seg_rows(cnt[p]);
        }
        soff[P] = o;
    }
    __syncthreads();
    for (int p = threadIdx.x; p <= P; p += blockDim.x) off[p] = soff[p];
    // 5. stable scatter: warp w walks chunks w, w + 32, ... in pair order
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    for (int c = warp; c < nchunks; c += blockDim.x / 32) {
        int32_t* base = scratch + c * P;
        for (int g = c * kPlanChunk; g < min(npairs, (c + 1) * kPlanChunk); g += 32) {
            const int i = g + lane;
            int p = i < npairs ? phys[i] : -1;
            if (p >= P || p < 0) {
                if (i < npairs) pos[i] = -1;          // an id outside [0, P) is left out of the plan
                p = -1;
            }
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, p);
            int before = 0;
            if (p >= 0) {
                before = base[p];
                pos[i] = soff[p] + before + __popc(peers & lt);
            }
            __syncwarp();
            if (p >= 0 && lane == __ffs(peers) - 1) base[p] = before + __popc(peers);
            __syncwarp();
        }
    }
}

// Device address of g_plan_scratch, looked up once per device and context:
// the address belongs to the module loaded into the device's current
// context, so when that context is created anew (after cudaDeviceReset, or
// once the primary context was released and retained again) the address is
// looked up again.  Contexts are told apart by the driver's context id, which
// is unique for the life of the process (a re-created context may reuse the
// old handle's value, never its id).
constexpr int kMaxDevices = 64;
struct ScratchAddr {
    unsigned long long ctx_id;
    void* addr;
};
ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

void* driver_fn(const char* name)
{
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return p;
}

// id of the context current on this thread; 0 when none is bound yet
bool current_ctx_id(unsigned long long* id)
{
    static CtxGetCurrentFn get_ctx = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent"));
    static CtxGetIdFn get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId"));
    *id = 0;
    if (!get_ctx || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return false;
    return !ctx || get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

extern "C" mm_status mm_plan_dispatch_static(const int32_t* phys, int64_t npairs, int num_physical, int32_t* pos,
                                             int32_t* offsets, mm_stream stream)
{
    if (npairs < 0 || num_physical < 1 || num_physical > MM_MAX_EXPERTS || !offsets || (npairs > 0 && (!phys || !pos)))
        return MM_ERR_INVALID_ARG;
    if (npairs > kPlanMaxPairs) return MM_ERR_CAPACITY;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MM_ERR_CUDA;
    }
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        unsigned long long id = 0;
        if (!current_ctx_id(&id)) return MM_ERR_CUDA;
        ScratchAddr& slot = g_scratch_addr[dev];
        if (!slot.addr || id == 0 || slot.ctx_id != id) {
            // set-up: the address of the array in the current context (this
            // also binds the device's primary context when none is yet)
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || !p) {
                cudaGetLastError();
                return MM_ERR_CUDA;
            }
            if (id == 0 && (!current_ctx_id(&id) || id == 0)) return MM_ERR_CUDA;
            slot.ctx_id = id;
            slot.addr = p;
        }
        scratch = slot.addr;
    }
    plan_kernel<<<1, kPlanThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        phys, static_cast<int>(npairs), num_physical, static_cast<int32_t*>(scratch), pos, offsets);
    if (cudaGetLastError() != cudaSuccess) return MM_ERR_CUDA;
    return MM_OK;
}
