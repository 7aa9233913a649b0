// mm_gemm16.cu -- the a16w4 variant's persistent grouped GEMM: bf16 token
// rows x MXFP4 expert weights.  The pages' serving arms without expert
// parallelism run the same MXFP4 routed experts with bf16 activations
// ("InferenceX PR #3430", draft-precision notes); routing, EPLB remap,
// dispatch and combine are the a8w4 path's.
//
// The block-scaled MMA kinds take only 8-, 6- and 4-bit operands, so bf16
// activations meet the weights in a kind::f16 MMA with both operands bf16.
// The weights are converted in registers and written to tensor memory, which
// is where a tcgen05 MMA may read its A operand from:
//
//   D[128 weight rows][N tokens] += A . B^T over K = 16 per MMA
//   A = 128 weight rows in bf16 in tensor memory (lane = row, two K elements
//       per 32-bit column), B = the token tile's bf16 rows in shared memory
//       (K-major, 128-byte swizzle), N = the tile's rows rounded up to 16
//       (at most 128), fp32 accumulators in tensor memory.
//
// Tokens sit on N, so a short tile costs a narrow MMA, and the shared-memory
// traffic of an MMA is the token rows alone.
//
//   GEMM1 unit (tile, j): I-columns i0 = 64 j .. +64.  A row 32q + l holds the
//       gate row i0 + 16q + l (l < 16) or the up row i0 + 16q + l - 16
//       (l >= 16), so one epilogue warp holds both factors of 16 I-columns and
//       pairs them with one shuffle; h = silu(gate) * up, rounded to bf16, is
//       stored as GEMM2's token operand.
//   GEMM2 unit (tile, mb): output features mb*128 .. +128.
//
// Warp roles (736 threads with 16 converter warps): 0 = weight producer (bulk copies of the packed
// weight rows and their scale tiles; it also draws the units), 1 = TMEM owner
// + MMA issuer, 2 = token producer (TMA for the token rows; a GEMM2 unit first
// waits, bounded, until the GEMM1 units of its tile have published h),
// 3..18 = converters (warp w: TMEM lane quarter w % 4, K quarter (w - 3) / 4
// of each 128-wide stage, i.e. one 32-element scale block), 19..22 = epilogue
// (lane quarter w % 4).  A converter warp's time per stage is a latency
// chain (shared-memory load, conversion, tensor-memory store), so there are
// four per scheduler, and a warp waits for its store of stage s only after it
// has converted stage s + 1.
// Three rings: packed weights (deep: the weight stream is what decode waits
// on, and a converter frees a slot as soon as it has read it), token rows
// (shallow: 32 KB a slot), and A slots in tensor memory between converters
// and MMA.  The accumulator is double-buffered.  Units are handed out at run
// time through a global counter and a ring in shared memory, GEMM1 units first.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

#ifndef MM_CONV_WARPS
#define MM_CONV_WARPS 16
#endif
constexpr int kConvWarps = MM_CONV_WARPS;                  // 8 or 16
static_assert(kConvWarps == 8 || kConvWarps == 16, "converter warps");
constexpr int kKParts = kConvWarps / 4;                    // K parts of a stage per lane quarter
constexpr int kEPT = 128 / kKParts;                        // elements a converter thread converts per stage
constexpr int kTokWarp = 2;
constexpr int kConvWarp0 = 3, kConvThreads = 32 * kConvWarps;
constexpr int kEpi16Warp0 = kConvWarp0 + kConvWarps, kEpi16Threads = 128;
constexpr int kT16Threads = 32 * kEpi16Warp0 + kEpi16Threads;
constexpr int kWRing = 12;                                 // packed-weight stages
constexpr int kTRing = 3;                                  // token stages
constexpr int kARing = 4;                                  // A slots in tensor memory
constexpr int kTokHalfBytes = 128 * 128;                   // 128 rows x 64 bf16: one swizzle column
constexpr int kTokStageBytes = 2 * kTokHalfBytes;          // K = 128 of up to 128 token rows
constexpr int kRawBytes = 8192;                            // packed e2m1 of a stage: 128 rows x 128 K
constexpr int kSf16Bytes = 1024;                           // one or two 512-byte scale tiles
constexpr int kWStageBytes = kRawBytes + kSf16Bytes;
constexpr int kURing16 = 4;
constexpr int kBar16Bytes = 512;
constexpr int kSmem16Bytes = kTRing * kTokStageBytes + kWRing * kWStageBytes + kBar16Bytes + 1024;
static_assert(kTokStageBytes % 1024 == 0 && kWStageBytes % 1024 == 0, "1024-byte aligned stages");
static_assert(kSmem16Bytes <= 232448, "shared memory per block");
// tensor memory: accumulators [0, 256) = 2 x 128 columns, A slots [256, 512) = 4 x 64
constexpr uint32_t kTmem16Cols = 512, kAcc16Cols = 128, kASlot0 = 256, kASlotCols = 64;

struct Smem16 {
    uint8_t* tok;       // [kTRing][kTokStageBytes]
    uint8_t* wst;       // [kWRing][kWStageBytes]
    uint64_t* wfull;    // [kWRing] weight bytes landed
    uint64_t* wempty;   // [kWRing] read by the 8 converter warps
    uint64_t* tfull_;   // [kTRing] token rows landed
    uint64_t* tempty_;  // [kTRing] the stage's MMAs finished
    uint64_t* afull;    // [kARing] A slot written by the 8 converter warps
    uint64_t* aempty;   // [kARing] the slot's MMAs finished
    uint64_t* dfull;    // [2] accumulator complete
    uint64_t* dempty;   // [2] accumulator drained by the epilogue
    uint64_t* ufull;    // [kURing16] unit slot written
    uint64_t* uempty;   // [kURing16] unit slot read by every consumer
    uint64_t* drain;    // the MMA thread's own wait for its issued work after an abort
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    volatile int* uring;
};

__device__ __forceinline__ Smem16 smem16(uint8_t* base)
{
    Smem16 s;
    s.tok = base;
    s.wst = base + kTRing * kTokStageBytes;
    uint64_t* b = reinterpret_cast<uint64_t*>(s.wst + kWRing * kWStageBytes);
    s.wfull = b;
    s.wempty = s.wfull + kWRing;
    s.tfull_ = s.wempty + kWRing;
    s.tempty_ = s.tfull_ + kTRing;
    s.afull = s.tempty_ + kTRing;
    s.aempty = s.afull + kARing;
    s.dfull = s.aempty + kARing;
    s.dempty = s.dfull + 2;
    s.ufull = s.dempty + 2;
    s.uempty = s.ufull + kURing16;
    s.drain = s.uempty + kURing16;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
    s.uring = s.abort_flag + 1;
    static_assert((2 * kWRing + 2 * kTRing + 2 * kARing + 4 + 2 * kURing16 + 1) * 8 + 8 + 4 * kURing16 <= kBar16Bytes,
                  "barrier block");
    return s;
}

// A ring position: slot and phase, advanced once per stage.
template <int N>
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance()
    {
        if (++slot == N) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

struct Unit16 {
    int phase;       // 1 or 2
    int tile;
    int expert;
    int row0, rows;
    int n;           // MMA N: rows rounded up to 16
    int tbox;        // token box map: 16 << tbox rows
    int ksteps;
    int sel;         // GEMM1: which 64-row half of the gate/up blocks; GEMM2: member of the W2 pair
    int col0;        // GEMM1: first I-column; GEMM2: first output feature
    int64_t wblk;    // weight block of stage 0 (a stage adds 2)
};

__device__ __forceinline__ bool decode16(const Gemm16Args& g, int u, Unit16& un)
{
    const int ntiles = *g.num_tiles;
    const int per1 = g.I / 64, per2 = g.H / 128;
    const int units1 = ntiles * per1, units2 = ntiles * per2;
    if (u < 0 || u >= units1 + units2) return false;
    int j;
    if (u < units1) {
        un.phase = 1;
        un.tile = u / per1;
        j = u % per1;
    } else {
        un.phase = 2;
        un.tile = (u - units1) / per2;
        j = (u - units1) % per2;
    }
    un.expert = g.tile_expert[un.tile];
    un.row0 = g.tile_row0[un.tile];
    un.rows = g.tile_rows[un.tile];
    if (!MM_CHECK(un.expert >= 0 && un.expert < g.P && un.row0 >= 0 && un.rows >= 1 && un.rows <= 128 &&
                      un.row0 + un.rows <= g.rows_cap,
                  g.status, kSiteGemmTile))
        return false;
    un.n = (un.rows + 15) & ~15;
    un.tbox = un.rows <= 16 ? 0 : (un.rows <= 32 ? 1 : (un.rows <= 64 ? 2 : 3));
    if (un.phase == 1) {
        // W1 group nb = j / 2 pairs gate block (member 0) and up block (member 1)
        un.sel = j % 2;
        un.col0 = 64 * j;
        un.ksteps = g.H / 128;
        un.wblk = (static_cast<int64_t>(un.expert) * (g.I / 128) + j / 2) * un.ksteps * 2;
    } else {
        // W2 group j / 2 pairs output rows [256 (j/2), +128) and [256 (j/2) + 128, +128)
        un.sel = j % 2;
        un.col0 = 128 * j;
        un.ksteps = g.I / 128;
        un.wblk = (static_cast<int64_t>(un.expert) * ((g.H + 255) / 256) + j / 2) * un.ksteps * 2 + un.sel;
    }
    return true;
}

using UQ = Ring<kURing16>;

__device__ __forceinline__ bool push16(const Gemm16Args& g, const Smem16& s, UQ& q, int& u)
{
    u = *s.abort_flag ? 0x7FFFFFFF : atomicAdd(g.unit_next, 1);
    if (!mbar_wait(&s.uempty[q.slot], q.phase ^ 1u, g.status, s.abort_flag, kSiteUnitQueue)) return false;
    s.uring[q.slot] = u;
    mbar_arrive(&s.ufull[q.slot]);
    q.advance();
    return true;
}

__device__ __forceinline__ bool pop16(const Gemm16Args& g, const Smem16& s, UQ& q, int& u)
{
    if (!mbar_wait(&s.ufull[q.slot], q.phase, g.status, s.abort_flag, kSiteUnitQueue)) return false;
    u = s.uring[q.slot];
    mbar_arrive(&s.uempty[q.slot]);
    q.advance();
    return true;
}

// ---- FP4 -> bf16 ---------------------------------------------------------------
// Bit placement: a nibble n = s|e1 e0|m spread so that e1 e0 m sit at bf16
// bits 8..6 and s at bit 15 reads, as a bf16 bit pattern, (e2m1 value) x
// 2^-126 (its exponent field lands in the low bits of the bf16 exponent, bias
// 1 against 127, and its subnormal 0.5 becomes the bf16 subnormal 2^-127).
// For an element pair, x0 (even element) in bits 0..3 and x1 in bits 16..19 of
// v, one multiply by 4160 = 2^12 + 2^6 adds v << 6 (magnitudes to 6..8 and
// 22..24) and v << 12 (signs to 15 and 31) without overlapping carries, and a
// mask keeps those eight bits.  One bf16 multiply by 2^(X + 126) then gives
// the element times its block scale 2^X exactly (two significant bits at
// most); for X + 126 > 127 the factor is split in two.
__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ __nv_bfloat162 bf16x2_pow2(int e)     // 2^e, -133 < e <= 127: normal range used
{
    const uint32_t b = static_cast<uint32_t>(e + 127) << 7;
    const uint32_t r = b | (b << 16);
    return *reinterpret_cast<const __nv_bfloat162*>(&r);
}

// 4 packed bytes (8 elements, element 2i in the low nibble of byte i) ->
// 4 bf16x2 words (element 2i in the low half), times f1.
__device__ __forceinline__ void e2m1x8_to_bf16x8(uint32_t w, __nv_bfloat162 f1, uint32_t* o)
{
    const uint32_t ev = w & 0x0F0F0F0Fu;            // even elements' nibbles
    const uint32_t od = (w >> 4) & 0x0F0F0F0Fu;     // odd elements' nibbles
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // byte 0 = even nibble j, byte 2 = odd nibble j; bytes 1 and 3 replicate
        // the sign bit of byte 0 of ev, which is 0 (a nibble is below 0x80)
        const uint32_t v = prmt_b32(ev, od, static_cast<uint32_t>(j) | 0x80u | ((4u + j) << 8) | 0x8000u);
        const uint32_t r = (v * 4160u) & 0x81C081C0u;
        __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&r);
        x = __hmul2(x, f1);
        o[j] = *reinterpret_cast<const uint32_t*>(&x);
    }
}

// 16 packed bytes (32 elements, one block with scale byte sb) -> 16 bf16x2 words.
__device__ __forceinline__ void convert32(const uint4 q, uint32_t sb_u, uint32_t* w)
{
    const int sb = static_cast<int>(sb_u);     // X = sb - 127
    const bool wide = sb >= 129;               // X + 126 > 127
    const __nv_bfloat162 f1 = bf16x2_pow2(wide ? 127 : sb - 1);
    e2m1x8_to_bf16x8(q.x, f1, w);
    e2m1x8_to_bf16x8(q.y, f1, w + 4);
    e2m1x8_to_bf16x8(q.z, f1, w + 8);
    e2m1x8_to_bf16x8(q.w, f1, w + 12);
    if (wide) {
        const __nv_bfloat162 f2 = bf16x2_pow2(sb - 128);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
            v = __hmul2(v, f2);
            w[i] = *reinterpret_cast<const uint32_t*>(&v);
        }
    }
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t* r)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] . B^T, bf16 operands, fp32 accumulate.
template <bool kAccumulate>
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc)
{
    if (kAccumulate)
        asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem), "r"(a_tmem),
                     "l"(bdesc), "r"(idesc)
                     : "memory");
    else
        asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 0;" ::"r"(d_tmem), "r"(a_tmem),
                     "l"(bdesc), "r"(idesc)
                     : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B bf16, both
// K-major, M = 128, N = n (multiple of 16, <= 256).
__device__ __forceinline__ uint32_t idesc_bf16(uint32_t n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ int ld_acquire_i32(const int* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ---- weight producer (warp 0, one thread): draws the units --------------------
__device__ __forceinline__ void wproducer16(const Gemm16Args& g, const Smem16& s)
{
    Ring<kWRing> w;
    int armed[kWRing];
    for (int i = 0; i < kWRing; ++i) armed[i] = -1;
    Unit16 un;
    UQ q;
    for (;;) {
        int u;
        if (!push16(g, s, q, u) || *s.abort_flag || !decode16(g, u, un)) break;
        const uint32_t bytes = kRawBytes + (un.phase == 1 ? 1024u : 512u);
        for (int ks = 0; ks < un.ksteps; ++ks) {
            if (!mbar_wait(&s.wempty[w.slot], w.phase ^ 1u, g.status, s.abort_flag, kSiteProducerEmpty)) break;
            uint8_t* raw = s.wst + w.slot * kWStageBytes;
            uint8_t* sf = raw + kRawBytes;
            mbar_arrive_expect_tx(&s.wfull[w.slot], bytes);
            armed[w.slot] = static_cast<int>(w.phase);
            const int64_t blk = un.wblk + 2 * ks;
            if (un.phase == 1) {
                // the unit's 64-row halves of the gate block and of the up block
                bulk_load(raw, g.w1 + blk * 8192 + un.sel * 4096, 4096, &s.wfull[w.slot]);
                bulk_load(raw + 4096, g.w1 + (blk + 1) * 8192 + un.sel * 4096, 4096, &s.wfull[w.slot]);
                bulk_load(sf, g.w1_sf + blk * 512, 1024, &s.wfull[w.slot]);
            } else {
                bulk_load(raw, g.w2 + blk * 8192, 8192, &s.wfull[w.slot]);
                bulk_load(sf, g.w2_sf + blk * 512, 512, &s.wfull[w.slot]);
            }
            w.advance();
        }
    }
    if (*s.abort_flag) {
        // let copies already in flight land before the CTA exits
        for (int i = 0; i < kWRing; ++i) {
            if (armed[i] < 0) continue;
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(&s.wfull[i], static_cast<uint32_t>(armed[i])))
                if (globaltimer() - t0 > kWaitLimitNs / 4) break;
        }
    }
}

// ---- token producer (warp 2, one thread) ------------------------------------------
__device__ __forceinline__ void tproducer16(const Gemm16Maps& maps, const Gemm16Args& g, const Smem16& s)
{
    const uint64_t pol_a = policy_evict_last();
    Ring<kTRing> t;
    int armed[kTRing];
    for (int i = 0; i < kTRing; ++i) armed[i] = -1;
    Unit16 un;
    UQ q;
    for (;;) {
        int u;
        if (!pop16(g, s, q, u) || *s.abort_flag || !decode16(g, u, un)) break;
        const CUtensorMap* tmap = un.phase == 1 ? &maps.xd[un.tbox] : &maps.hb[un.tbox];
        if (un.phase == 2) {
            const int need = g.I / 64 + (g.fault == kFaultGemmDependency ? 1 : 0);
            if (ld_acquire_i32(&g.done1[un.tile]) < need) {
                const uint64_t t0 = globaltimer();
                while (ld_acquire_i32(&g.done1[un.tile]) < need) {
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
        const uint32_t bytes = 2u * (16u << un.tbox) * 128u;
        for (int ks = 0; ks < un.ksteps; ++ks) {
            if (!mbar_wait(&s.tempty_[t.slot], t.phase ^ 1u, g.status, s.abort_flag, kSiteProducerEmpty)) break;
            uint8_t* st = s.tok + t.slot * kTokStageBytes;
            mbar_arrive_expect_tx(&s.tfull_[t.slot], bytes);
            armed[t.slot] = static_cast<int>(t.phase);
            tma_load_2d(st, tmap, ks * 128, un.row0, &s.tfull_[t.slot], pol_a);
            tma_load_2d(st + kTokHalfBytes, tmap, ks * 128 + 64, un.row0, &s.tfull_[t.slot], pol_a);
            t.advance();
        }
    }
    if (*s.abort_flag) {
        for (int i = 0; i < kTRing; ++i) {
            if (armed[i] < 0) continue;
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(&s.tfull_[i], static_cast<uint32_t>(armed[i])))
                if (globaltimer() - t0 > kWaitLimitNs / 4) break;
        }
    }
}

// ---- MMA issuer (warp 1, all lanes) ------------------------------------------
// The whole warp runs the loop, so every operand of an MMA is computed
// warp-uniformly; one elected lane issues the tensor-core instructions.  (An
// MMA of small N is issued in a few tens of cycles; the issuing thread's own
// operand arithmetic is what would otherwise set the rate.)
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

__device__ __forceinline__ bool pop16_warp(const Gemm16Args& g, const Smem16& s, UQ& q, int& u)
{
    const bool ok = mbar_wait(&s.ufull[q.slot], q.phase, g.status, s.abort_flag, kSiteUnitQueue);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    u = s.uring[q.slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&s.uempty[q.slot]);
    q.advance();
    return true;
}

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const Gemm16Args& g, const Smem16& s,
                                          int site)
{
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, g.status, s.abort_flag, site));
}

__device__ __forceinline__ void mma16(const Gemm16Args& g, const Smem16& s, uint32_t tmem)
{
    static_assert(kTRing * kTokStageBytes + 1024 < (1 << 18), "descriptor address field");
    const uint64_t b_desc0 = desc_kmajor_sw128(s.tok);
    constexpr uint64_t kStageDesc = kTokStageBytes >> 4, kHalfDesc = kTokHalfBytes >> 4;
    Ring<kTRing> t;
    Ring<kARing> a;
    int acc = 0;       // accumulators used so far: buffer acc & 1, phase (acc >> 1) & 1
    bool aborted = false;
    Unit16 un;
    UQ q;
    for (;;) {
        int u;
        if (!pop16_warp(g, s, q, u) || *s.abort_flag || !decode16(g, u, un)) break;
        const int buf = acc & 1;
        const uint32_t aph = static_cast<uint32_t>(acc >> 1) & 1u;
        if (!wait_warp(&s.dempty[buf], aph ^ 1u, g, s, kSiteMmaTmemEmpty)) {
            aborted = true;
            break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(buf) * kAcc16Cols;
        const uint32_t id = idesc_bf16(static_cast<uint32_t>(un.n));
        for (int ks = 0; ks < un.ksteps; ++ks) {
            // this stage's token rows (TMA) and A slot (converters)
            if (!wait_warp(&s.tfull_[t.slot], t.phase, g, s, kSiteMmaFull) ||
                !wait_warp(&s.afull[a.slot], a.phase, g, s, kSiteMmaFull)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint64_t bd = b_desc0 + static_cast<uint64_t>(t.slot) * kStageDesc;
            const uint32_t at = tmem + kASlot0 + static_cast<uint32_t>(a.slot) * kASlotCols;
            if (elect_one()) {
                // K = 128: eight MMAs of K = 16; the token rows' K halves are two swizzle columns
                if (ks == 0)
                    mma_bf16_tmem_a<false>(d, at, bd, id);
                else
                    mma_bf16_tmem_a<true>(d, at, bd, id);
                mma_bf16_tmem_a<true>(d, at + 8, bd + 2, id);
                mma_bf16_tmem_a<true>(d, at + 16, bd + 4, id);
                mma_bf16_tmem_a<true>(d, at + 24, bd + 6, id);
                mma_bf16_tmem_a<true>(d, at + 32, bd + kHalfDesc, id);
                mma_bf16_tmem_a<true>(d, at + 40, bd + kHalfDesc + 2, id);
                mma_bf16_tmem_a<true>(d, at + 48, bd + kHalfDesc + 4, id);
                mma_bf16_tmem_a<true>(d, at + 56, bd + kHalfDesc + 6, id);
                tc_commit(&s.tempty_[t.slot]);
                tc_commit(&s.aempty[a.slot]);
            }
            __syncwarp();
            t.advance();
            a.advance();
        }
        if (aborted || *s.abort_flag) break;
        if (elect_one()) tc_commit(&s.dfull[buf]);
        __syncwarp();
        ++acc;
    }
    if (*s.abort_flag) {
        // drain issued tensor-core work before the allocation is freed, on a
        // barrier no other role waits on
        if (elect_one()) {
            tc_commit(s.drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(s.drain, 0))
                if (globaltimer() - t0 > kWaitLimitNs / 4) break;
        }
        __syncwarp();
    }
}

// ---- converters: warps 3..18 -----------------------------------------------------
// Thread (quarter qd, lane l) writes A row r = 32 qd + l; its warp covers the
// K quarter kq (32 elements, one scale block) of every stage.  A weight slot
// is released once the warp has converted what it read; the tensor-memory
// store of stage s is waited for (and its A slot published) after stage s + 1
// is converted, and at the end of every unit.
__device__ __forceinline__ void convert16(const Gemm16Args& g, const Smem16& s, uint32_t tmem)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qd = warp & 3, kq = (warp - kConvWarp0) >> 2;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * qd) << 16) + kASlot0 + (kEPT / 2u) * kq;
    Ring<kWRing> w;
    Ring<kARing> a;
    int pending = -1;          // A slot whose store is in flight
    Unit16 un;
    UQ q;
    auto publish = [&]() {
        if (pending >= 0) {
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.afull[pending]);
            pending = -1;
        }
    };
    for (;;) {
        int u;
        if (!pop16(g, s, q, u) || *s.abort_flag || !decode16(g, u, un)) break;
        // source row of this thread's A row in the stage's packed weights and scale tiles
        int src, sfrow, sftile;
        if (un.phase == 1) {
            const bool up = lane >= 16;
            const int i = 16 * qd + (lane & 15);            // row within the unit's 64 I-columns
            src = (up ? 4096 : 0) + i * 64;
            sfrow = 64 * un.sel + i;                         // row within the 128-row block
            sftile = up ? 512 : 0;
        } else {
            const int r = 32 * qd + lane;
            src = r * 64;
            sfrow = r;
            sftile = 0;
        }
        src += (kEPT / 2) * kq;
        const int sfo = kRawBytes + sftile + (sfrow % 32) * 16 + (sfrow / 32) * 4 + (kEPT / 32) * kq;
        bool ok = true;
        for (int ks = 0; ks < un.ksteps; ++ks) {
            // warp-uniform decisions: after an abort the producers still let
            // copies in flight land, so lanes could otherwise disagree before
            // the warp-collective tensor-memory store
            ok = mbar_wait(&s.wfull[w.slot], w.phase, g.status, s.abort_flag, kSiteMmaFull);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                ok = false;
                break;
            }
            const uint8_t* raw = s.wst + w.slot * kWStageBytes;
            uint32_t cw[kEPT / 2];
#pragma unroll
            for (int b = 0; b < kEPT / 32; ++b) {
                const uint4 pk = reinterpret_cast<const uint4*>(raw + src)[b];
                convert32(pk, raw[sfo + b], cw + 16 * b);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.wempty[w.slot]);
            w.advance();
            publish();
            ok = mbar_wait(&s.aempty[a.slot], a.phase ^ 1u, g.status, s.abort_flag, kSiteMmaTmemEmpty);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if constexpr (kEPT == 32)
                tmem_st_32x32b_x16(lane_addr + static_cast<uint32_t>(a.slot) * kASlotCols, cw);
            else
                tmem_st_32x32b_x32(lane_addr + static_cast<uint32_t>(a.slot) * kASlotCols, cw);
            pending = a.slot;
            a.advance();
        }
        if (ok) publish();
        if (!ok || *s.abort_flag) break;
    }
    if (pending >= 0) tmem_st_wait();    // no store may be left in flight when the CTA tears down
}

// 16 consecutive accumulator columns of this warp's 32 rows
__device__ __forceinline__ void ld16_16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    tmem_ld_32x32b_x16(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- epilogue: warps 10..13 -------------------------------------------------------
__device__ __forceinline__ void epilogue16(const Gemm16Args& g, const Smem16& s, uint32_t tmem)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qd = warp & 3;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    int acc = 0;
    Unit16 un;
    UQ q;
    for (;;) {
        int u;
        if (!pop16(g, s, q, u) || *s.abort_flag || !decode16(g, u, un)) break;
        const int buf = acc & 1;
        if (!mbar_wait(&s.dfull[buf], static_cast<uint32_t>(acc >> 1) & 1u, g.status, s.abort_flag,
                       kSiteEpiTmemFull))
            break;
        tc_fence_after();
        const uint32_t base = lane_addr + static_cast<uint32_t>(buf) * kAcc16Cols;
        for (int c0 = 0; c0 < un.n; c0 += 16) {
            float v[16];
            ld16_16(base + c0, v);
            if (un.phase == 1) {
                // lanes l and l + 16 hold gate and up of I-column col0 + 16 qd + l
                const int col = un.col0 + 16 * qd + (lane & 15);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float upv = __shfl_down_sync(0xFFFFFFFFu, v[i], 16);
                    const int r = c0 + i;
                    if (lane < 16 && r < un.rows) {
                        const float gv = v[i];
                        const float h = gv / (1.0f + __expf(-gv)) * upv;
                        g.hb[static_cast<int64_t>(un.row0 + r) * g.I + col] = __float2bfloat16_rn(h);
                    }
                }
            } else {
                const int col = un.col0 + 32 * qd + lane;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = c0 + i;
                    if (r < un.rows) g.y[static_cast<int64_t>(un.row0 + r) * g.H + col] = __float2bfloat16_rn(v[i]);
                }
            }
        }
        tc_fence_before();
        mbar_arrive(&s.dempty[buf]);
        if (un.phase == 1) {
            // publish this unit's share of hb for the tile's GEMM2 units
            fence_proxy_async_global();
            __threadfence();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (threadIdx.x == kEpi16Warp0 * 32) atomicAdd(&g.done1[un.tile], 1);
        }
        ++acc;
    }
}

__global__ void __launch_bounds__(kT16Threads, 1)
    gemm16_kernel(const __grid_constant__ Gemm16Maps maps, const __grid_constant__ Gemm16Args g)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Smem16 s = smem16(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kWRing; ++i) {
            mbar_init(&s.wfull[i], 1);
            mbar_init(&s.wempty[i], kConvThreads / 32);
        }
        for (int i = 0; i < kTRing; ++i) {
            mbar_init(&s.tfull_[i], 1);
            mbar_init(&s.tempty_[i], 1);
        }
        for (int i = 0; i < kARing; ++i) {
            mbar_init(&s.afull[i], kConvThreads / 32);
            mbar_init(&s.aempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.dfull[i], 1);
            mbar_init(&s.dempty[i], kEpi16Threads);
        }
        for (int i = 0; i < kURing16; ++i) {
            mbar_init(&s.ufull[i], 1);
            // consumers: token producer, MMA thread, converters, epilogue
            mbar_init(&s.uempty[i], 2 + kConvThreads + kEpi16Threads);
        }
        mbar_init(s.drain, 1);
        *s.abort_flag = 0;
        fence_mbar_init();
        for (int i = 0; i < kTokBoxes; ++i) {
            prefetch_tmap(&maps.xd[i]);
            prefetch_tmap(&maps.hb[i]);
        }
    }
    if (warp == 1) {
        tmem_alloc(s.tmem_slot, kTmem16Cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s.tmem_slot;
    if (warp == 0) {
        if (lane == 0) wproducer16(g, s);
    } else if (warp == 1) {
        mma16(g, s, tmem);
    } else if (warp == kTokWarp) {
        if (lane == 0) tproducer16(maps, g, s);
    } else if (warp < kEpi16Warp0) {
        convert16(g, s, tmem);
    } else {
        epilogue16(g, s, tmem);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmem16Cols);
    }
}

}  // namespace

cudaError_t gemm16_prepare()
{
    return cudaFuncSetAttribute(gemm16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem16Bytes);
}

cudaError_t launch_gemm16(const mm_ctx* c, cudaStream_t s)
{
    Gemm16Args g;
    g.w1 = c->w1;
    g.w1_sf = c->w1_sf;
    g.w2 = c->w2;
    g.w2_sf = c->w2_sf;
    g.hb = reinterpret_cast<__nv_bfloat16*>(c->hq);
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
    g.fault = c->fault;
    g.P = wexp(c);
    g.rows_cap = static_cast<int>(c->rows_cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c->sms));
    cfg.blockDim = dim3(kT16Threads);
    cfg.dynamicSmemBytes = kSmem16Bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm16_kernel, c->maps16, g);
}

}  // namespace mm
