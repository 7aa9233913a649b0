// mm_gemm.cu -- the large-input path's persistent grouped GEMM kernel: GEMM1
// (+SwiGLU, MXFP8 requant) and GEMM2 units over the token tiles that the
// permute kernels wrote to global memory.  The machinery lives in mm_gemm.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mm_gemm.cuh"

namespace mm {
namespace {

using Geo = GeomLarge;
constexpr int kSmemBytes = Geo::kSmemBytes + 1024;

__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs g)
{
    // the batch went to the pair kernel (launched after this one): every CTA
    // reads the same choice and returns before touching anything
    if (g.select == 1 && g.num_tiles[3] != 0) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const GemmSmem s = gemm_smem(smem, smem + Geo::kStageRegion);
    const uint32_t tmem = gemm_setup<Geo>(s, maps);
    TileView tv;
    tv.expert = g.tile_expert;
    tv.row0 = g.tile_row0;
    tv.rows = g.tile_rows;
    tv.ntiles = *g.num_tiles;
    gemm_roles<Geo>(maps, g, tv, s, tmem);
    gemm_teardown(tmem);
}

}  // namespace

cudaError_t gemm_prepare(int dev)
{
    (void)dev;
    return cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

void fill_gemm_args(const mm_ctx* c, GemmArgs* gp)
{
    GemmArgs& g = *gp;
    g.w1 = c->w1;
    g.w2 = c->w2;
    g.w1_sf = c->w1_sf;
    g.w2_sf = c->w2_sf;
    g.xs_t = c->xs_t;
    g.hq = c->hq;
    g.hs_t = c->hs_t;
    g.y = c->y;
    g.tile_expert = c->tile_expert;
    g.tile_row0 = c->tile_row0;
    g.tile_rows = c->tile_rows;
    g.num_tiles = c->num_tiles;
    g.done1 = c->done1;
    g.unit_next = c->unit_next;
    g.status = c->status;
    g.H = c->H;
    g.I = c->I;
    g.P = wexp(c);
    g.phases = 3;
    g.fault = c->fault;
    g.rows_cap = static_cast<int>(c->rows_cap);
    g.st_tile = c->st_tile;
    g.keep_weights = 0;
    g.select = 0;
}

cudaError_t launch_gemm(const mm_ctx* c, int64_t T, cudaStream_t s)
{
    (void)T;
    const bool pairs = gemm2_usable(c);
    if (pairs && c->gemm_2sm == 1) return launch_gemm2(c, s, 0);
    GemmArgs g;
    fill_gemm_args(c, &g);
    g.select = pairs ? 1 : 0;       // gemm_2sm == 2: the tile scan chooses on the device
    // Large batches give an expert several token tiles, each re-reading the
    // expert's weight blocks: loading them with the normal L2 policy rather
    // than evict-first measured 2% faster on the skewed 16384-token layer (its
    // hot experts have tens of tiles) and the same on uniform prefill.
    g.keep_weights = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c->sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_kernel, c->maps, g);
    if (e != cudaSuccess || !pairs) return e;
    return launch_gemm2(c, s, 2);
}

int gemm_kind(const mm_ctx* c)
{
    if (!gemm2_usable(c)) return 1;
    return c->gemm_2sm == 1 ? 2 : 4;
}

}  // namespace mm
