// mm_device.cuh -- sm_103a device helpers: mbarriers, TMA, tcgen05 (TMEM,
// block-scaled MMA), bounded waits and the element-format conversions used
// by the fused MoE kernels.  Inline PTX only; no library headers beyond the
// CUDA runtime's own.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp8.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mm_internal.h"

namespace mm {

// ---------------------------------------------------------------------------
// status latch and bounded waits
// ---------------------------------------------------------------------------
// Every spin-wait gives up after a bounded time of %globaltimer and latches
// MM_ERR_TIMEOUT with its site; kernels then drain and return instead of
// hanging.  Waits on progress made elsewhere (grid barriers, GEMM1 -> GEMM2
// dependencies) give up first; waits inside a CTA's own pipeline (mbarriers)
// get twice as long, so that the site reported is the root cause and not a
// stage starved by it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;          // 2 s: external progress
constexpr uint64_t kPipeWaitLimitNs = 2 * kWaitLimitNs;   // 4 s: own pipeline

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// status[0] = first error code, status[1] = the site that raised it
__device__ __forceinline__ void latch_error(int* status, int code, int site = 0)
{
    if (atomicCAS(status, 0, code) == 0) atomicExch(status + 1, site);
}

// Bounds checks of debug builds (compiled with MM_DEBUG): MM_CHECK(cond,
// status, site) is cond, and when cond is false it latches MM_ERR_DEVICE
// with the site, so the caller skips the access it guards.  In release builds
// it is the constant true and every check compiles away.
#ifdef MM_DEBUG
__device__ __forceinline__ bool debug_check(bool ok, int* status, int site)
{
    if (!ok) latch_error(status, MM_ERR_DEVICE, site);
    return ok;
}
#define MM_CHECK(cond, status, site) (::mm::debug_check((cond), (status), (site)))
#else
#define MM_CHECK(cond, status, site) true
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false on timeout
// (then MM_ERR_TIMEOUT is latched and *abort set so the caller unwinds).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, volatile int* abort,
                                          int site)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (globaltimer() - t0 > kPipeWaitLimitNs) {
            latch_error(status, MM_ERR_TIMEOUT, site);
            *abort = 1;
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------------------
// TMA and bulk copies (global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                            uint64_t* bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------------------
// thread-block clusters: rank, peer shared memory, cluster-wide barrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_peer_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// arrive (release at cluster scope) on an mbarrier of another CTA of the cluster
__device__ __forceinline__ void mbar_arrive_peer(uint32_t addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// Relaxed: orders nothing before it.  For signals whose only precondition is
// already complete in the signalling thread (a tensor-memory read followed by
// tcgen05.wait::ld); the release form measured ~1,000 cycles a call here.
__device__ __forceinline__ void mbar_arrive_peer_relaxed(uint32_t addr)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// try_wait with acquire at cluster scope (for arrivals made by another CTA)
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait as mbar_wait, with acquire at cluster scope.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int* status, volatile int* abort,
                                                  int site)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (*abort) return false;
        if (globaltimer() - t0 > kPipeWaitLimitNs) {
            latch_error(status, MM_ERR_TIMEOUT, site);
            *abort = 1;
            return false;
        }
    }
    return true;
}

// every thread of every CTA of the cluster
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Tile loads into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (`bar` a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* tmap, int32_t x, int32_t y, uint32_t bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(void* dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                                 uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// Ask for global bytes to be brought into L2 (no completion, no destination).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// generic-proxy global writes <-> async-proxy (TMA) global reads
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, block-scaled MMA, scale-factor copies, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= (A * SFA) . (B * SFB)^T ; A and B K-major in shared memory,
// one e8m0 scale per 32 along K read from tensor memory.
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// The same MMA with a compile-time accumulate flag: no predicate to compute
// in the issuing thread.  The issuing thread's own instruction count per MMA
// sets the MMA rate when the operands are small, so the K loop keeps to this form.
template <bool kAccumulate>
__device__ __forceinline__ void mma_mxf8f6f4_c(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t sfa_tmem, uint32_t sfb_tmem)
{
    if (kAccumulate)
        asm volatile(
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], 1;" ::"r"(
                d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
    else
        asm volatile(
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], 0;" ::"r"(
                d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
}

// Arrive on an mbarrier once every prior tcgen05 operation of this thread completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// ---- the 2-SM forms (cta_group::2): a CTA pair of a cluster works as one
// MMA.  Tensor memory is allocated collectively (one warp in each CTA, the
// same columns in both); the even CTA issues the MMAs, which take A's M rows
// half from each CTA's shared memory (its 128 rows of D in its own tensor
// memory) and B's N rows half from each; the block scales of A are each CTA's
// own rows', those of B cover all N in both CTAs' tensor memory; a scale copy
// issued by the even CTA moves each CTA's shared memory into its own tensor
// memory.  A kernel uses only one cta_group.
__device__ __forceinline__ void tmem_alloc2(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish2()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

template <bool kAccumulate>
__device__ __forceinline__ void mma2_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem)
{
    if (kAccumulate)
        asm volatile(
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], 1;" ::"r"(
                d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
    else
        asm volatile(
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], 0;" ::"r"(
                d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
}

// arrive on the mbarrier at this offset in each CTA of cta_mask once the
// pair's prior tcgen05 operations have completed
__device__ __forceinline__ void tc_commit2_mc(uint64_t* bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

__device__ __forceinline__ void tc_cp2_32x128b_x4(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 32 rows x 128 bits of shared memory into tensor memory, replicated into all
// four 32-lane quarters (the scale-factor layout the block-scaled MMA reads).
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (16-byte units), version 1, swizzle mode.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= static_cast<uint64_t>(swizzle & 7u) << 61;
    return d;
}
constexpr uint32_t kSwizzleNone = 0, kSwizzle128B = 2;

// K-major operand, 128-byte rows, 128-byte swizzle: 8-row atoms of 1024 B.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(const void* tile)
{
    return smem_desc(smem_u32(tile), 16, 1024, kSwizzle128B);
}

// 32 x 16-byte scale-factor block, no swizzle, 8-row core matrices 128 B apart.
__device__ __forceinline__ uint64_t desc_sf(const void* sf)
{
    return smem_desc(smem_u32(sf), 0, 128, kSwizzleNone);
}

// Instruction descriptor, block-scaled kinds: A = e4m3 (format 0), B = e2m1
// (format 5), e8m0 scales, both K-major, M = 128, N = n (multiple of 16, <= 256);
// sf_id picks the scale byte (the 32-wide K block) inside each scale column.
__device__ __forceinline__ uint32_t idesc_e4m3_e2m1(uint32_t n, uint32_t sf_id, uint32_t m = 128)
{
    uint32_t d = 0;
    d |= (sf_id & 3u) << 4;       // B scale-factor byte
    d |= 0u << 7;                 // A format: e4m3
    d |= 5u << 10;                // B format: e2m1
    d |= (n >> 3) << 17;          // N / 8
    d |= 1u << 23;                // scale format: ue8m0
    d |= (m >> 4) << 24;          // M / 16 (256 for a CTA pair)
    d |= (sf_id & 3u) << 29;      // A scale-factor byte
    return d;
}

// ---------------------------------------------------------------------------
// element formats
// ---------------------------------------------------------------------------
// floor(log2(a)) for finite a > 0 (normal or subnormal binary32)
__device__ __forceinline__ int floor_log2_f32(float a)
{
    const uint32_t b = __float_as_uint(a);
    const int ex = static_cast<int>((b >> 23) & 0xFFu);
    if (ex != 0) return ex - 127;
    return (31 - __clz(static_cast<int>(b & 0x7FFFFFu))) - 149;
}

// MX scale exponent for e4m3 elements: X = clamp(floor(log2 amax) - 8, -127, 127);
// amax == 0 -> -127.  Returns X; the stored scale byte is X + 127.
__device__ __forceinline__ int mx_e4m3_exponent(float amax)
{
    if (!(amax > 0.0f)) return -127;
    int x = floor_log2_f32(amax) - 8;
    return x < -127 ? -127 : (x > 127 ? 127 : x);
}

// 2^e as binary32 for e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// e4m3 code of v * 2^-X, nearest-even, saturating at 448; the sign is taken
// from v so that values that vanish keep it.
__device__ __forceinline__ uint32_t e4m3_code(float v, float inv_scale)
{
    const float a = __fmul_rn(fabsf(v), inv_scale);
    const uint32_t c = static_cast<uint32_t>(__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3)) & 0x7Fu;
    return c | ((__float_as_uint(v) >> 24) & 0x80u);
}

}  // namespace mm
