// mm_stages.cuh -- per-item bodies of the SIMT stages of the fused MoE
// forward (route one token, quantise + dispatch one 32-element block, combine
// one 8-element output chunk).  The standalone kernels and the fused
// small-input kernel call the same bodies.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "mm_device.cuh"
#include "mm_internal.h"

namespace mm {

// ---------------------------------------------------------------------------
// routing score: a fixed binary32 operation sequence (Cody-Waite reduction
// with a two-part ln 2, degree-7 Taylor polynomial in Horner form, 2^n by the
// exponent field), every step one IEEE-rounded add, mul or div and no fused
// multiply-add, so the score -- and with it the selected experts -- is the
// same on every machine that evaluates this sequence.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float exp_spec(float y)
{
    const float log2e = __uint_as_float(0x3FB8AA3Bu);
    const float ln2_hi = __uint_as_float(0x3F317200u);
    const float ln2_lo = __uint_as_float(0x35BFBE8Eu);
    const float c2 = __uint_as_float(0x3F000000u);  // 1/2
    const float c3 = __uint_as_float(0x3E2AAAABu);  // 1/6
    const float c4 = __uint_as_float(0x3D2AAAABu);  // 1/24
    const float c5 = __uint_as_float(0x3C088889u);  // 1/120
    const float c6 = __uint_as_float(0x3AB60B61u);  // 1/720
    const float c7 = __uint_as_float(0x39500D01u);  // 1/5040
    y = fminf(fmaxf(y, -87.0f), 88.0f);
    const float n = rintf(__fmul_rn(y, log2e));
    float r = __fsub_rn(y, __fmul_rn(n, ln2_hi));
    r = __fsub_rn(r, __fmul_rn(n, ln2_lo));
    float p = c7;
    p = __fadd_rn(__fmul_rn(p, r), c6);
    p = __fadd_rn(__fmul_rn(p, r), c5);
    p = __fadd_rn(__fmul_rn(p, r), c4);
    p = __fadd_rn(__fmul_rn(p, r), c3);
    p = __fadd_rn(__fmul_rn(p, r), c2);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    return __fmul_rn(p, exp2i(static_cast<int>(n)));
}

__device__ __forceinline__ float sigmoid_spec(float x)
{
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp_spec(-x)));
}

struct RouteArgs {
    const float* logits;   // [T, E]
    const float* bias;     // [E] or null
    const int32_t* map;    // [E, R]
    const int32_t* rc;     // [E]
    int32_t* idx;          // [T, k + ns]
    float* w;              // [T, k + ns]
    int32_t* phys;         // [T, k + ns]
    int64_t* counts;       // [E] of the bound layer, or null when not recording
    int64_t T;
    int E, k, R;
    int ns, P;             // fused shared experts: slot k + s -> physical P + s, weight 1
    int* status;           // latched device status (bounds checks of debug builds)
};

// Order-preserving map of a binary32 key to uint32 (larger key, larger code).
// Routing keys are sigmoid scores plus a finite bias: never NaN or -0, so
// equal codes are exactly equal keys.
__device__ __forceinline__ uint32_t key_code(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp routes token t: lane l holds experts l, l+32, ...  Each lane keeps
// the best of its own remaining experts; a round takes the warp maximum of
// those keys and, among the lanes that hold it, the lowest expert index (ties
// go to the lower expert), so k rounds select the experts in order.  Lane j
// keeps the j-th selection; lanes 0..k-1 write idx/w/phys and count the
// selections into shared memory (hist != null) or the global table; lanes
// k..k+ns-1 write the token's fused shared-expert slots (logical id E + s,
// weight 1, physical P + s), which are never counted.
template <int VPL>
__device__ __forceinline__ void route_token(const RouteArgs& a, int64_t t, int lane, int* hist)
{
    float s[VPL];
    uint32_t code[VPL];
    uint32_t avail = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        s[i] = 0.0f;
        code[i] = 0u;
        if (e < a.E) {
            s[i] = sigmoid_spec(a.logits[t * a.E + e]);
            code[i] = key_code(__fadd_rn(s[i], a.bias ? a.bias[e] : 0.0f));
            avail |= 1u << i;
        }
    }
    // this lane's best remaining expert: code, slot i, score
    uint32_t lc = 0u;
    int li = -1;
    float ls = 0.0f;
    auto local_best = [&]() {
        lc = 0u;
        li = -1;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (((avail >> i) & 1u) && (li < 0 || code[i] > lc)) {
                lc = code[i];
                li = i;
                ls = s[i];
            }
        }
    };
    local_best();
    int my_e = 0;
    float my_s = 0.0f;
#pragma unroll
    for (int j = 0; j < MM_MAX_TOPK; ++j) {
        if (j >= a.k) break;
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, li >= 0 ? lc : 0u);
        const uint32_t cand = (li >= 0 && lc == m) ? static_cast<uint32_t>(lane + 32 * li) : 0xFFFFFFFFu;
        const int be = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, cand));
        const float bs = __shfl_sync(0xFFFFFFFFu, ls, be & 31);
        if (lane == j) {
            my_e = be;
            my_s = bs;
        }
        if ((be & 31) == lane) {
            avail &= ~(1u << (be >> 5));
            local_best();
        }
    }
    // sum of the selected scores in selection order (the same in every lane)
    float S = __shfl_sync(0xFFFFFFFFu, my_s, 0);
    for (int j = 1; j < a.k; ++j) S = __fadd_rn(S, __shfl_sync(0xFFFFFFFFu, my_s, j));
    const int kk = a.k + a.ns;
    if (lane < a.k) {
        const int e = my_e;
        const int rc = a.rc[e];
        int p = -1;
        if (MM_CHECK(rc >= 1 && rc <= a.R, a.status, kSiteRouteMap)) {
            const uint32_t slot = static_cast<uint32_t>(t + lane) % static_cast<uint32_t>(rc);
            p = a.map[e * a.R + static_cast<int>(slot)];
        }
        // a map entry outside [0, P) is recorded and replaced by -1, which
        // every later stage of a debug build leaves out
        if (!MM_CHECK(p >= 0 && p < a.P, a.status, kSiteRouteMap)) p = -1;
        a.idx[t * kk + lane] = e;
        a.w[t * kk + lane] = __fdiv_rn(my_s, S);
        a.phys[t * kk + lane] = p;
        if (a.counts) {
            if (hist) atomicAdd(&hist[e], 1);
            else atomicAdd(reinterpret_cast<unsigned long long*>(a.counts + e), 1ull);
        }
    } else if (lane < kk) {
        const int sh = lane - a.k;
        a.idx[t * kk + lane] = a.E + sh;
        a.w[t * kk + lane] = 1.0f;
        a.phys[t * kk + lane] = a.P + sh;
    }
}

__device__ __forceinline__ void route_token_any(const RouteArgs& a, int64_t t, int lane, int* hist)
{
    const int vpl = (a.E + 31) / 32;
    if (vpl <= 4) route_token<4>(a, t, lane, hist);
    else if (vpl <= 8) route_token<8>(a, t, lane, hist);
    else route_token<16>(a, t, lane, hist);
}

// The bounds of a debug build's checks (unused otherwise).
struct DispatchBounds {
    int P;              // physical experts with weights
    int64_t rows_cap;   // dispatch rows reserved
    int* status;
};

// MXFP8 quantisation of block b (32 elements) of token t: 4 x 128-bit loads;
// the 32 e4m3 codes packed four to a word, and the e8m0 scale byte as the
// return value.
__device__ __forceinline__ uint8_t quant_block32(const __nv_bfloat16* __restrict__ x, int64_t t, int b, int H,
                                                uint32_t (&packed)[8])
{
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H + b * 32);
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 u = __ldg(src + q);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[q * 8 + 2 * i] = __uint_as_float(w4[i] << 16);
            v[q * 8 + 2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int X = mx_e4m3_exponent(amax);
    const float inv = exp2i(-X);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t wd = 0;
        if (amax > 0.0f) {
#pragma unroll
            for (int j = 0; j < 4; ++j) wd |= e4m3_code(v[4 * i + j], inv) << (8 * j);
        }
        packed[i] = wd;
    }
    return static_cast<uint8_t>(X + 127);
}

// MXFP8 quantisation of block b of token t and its dispatch to the token's k
// rows: 32 e4m3 codes per row (2 x 128-bit stores).  pos_t / phys_t: the k
// dispatch rows and physical experts of token t; off / toff: segment start row
// and first token tile of each expert (global or shared memory), which place
// the scale byte in the scale tile of the row's token tile.
// Callers map four consecutive lanes (lane % 4 == b % 4) to the four blocks of
// one 128-wide K chunk of one token, all four active together: their scale
// bytes are adjacent in the scale tile, so the first lane of the four stores
// them as one word instead of four byte stores.
__device__ __forceinline__ void quant_dispatch_block(const __nv_bfloat16* __restrict__ x, int64_t t, int b, int H,
                                                     int k, const int32_t* pos_t, const int32_t* phys_t,
                                                     const int32_t* off, const int32_t* toff, int tile,
                                                     uint8_t* __restrict__ xq, uint8_t* __restrict__ xs_t,
                                                     const DispatchBounds& chk)
{
    (void)chk;
    uint32_t packed[8];
    const uint32_t sbyte = quant_block32(x, t, b, H, packed);
    const int lane = threadIdx.x & 31;
    const unsigned group = 0xFu << (lane & ~3);
    uint32_t sword = sbyte;
    sword |= __shfl_down_sync(group, sbyte, 1, 4) << 8;
    sword |= __shfl_down_sync(group, sbyte, 2, 4) << 16;
    sword |= __shfl_down_sync(group, sbyte, 3, 4) << 24;
    const int kchunks = H / 128;
    for (int j = 0; j < k; ++j) {
        const int64_t row = pos_t[j];
        const int p = phys_t[j];
        if (!MM_CHECK(p >= 0 && p < chk.P && row >= 0 && row < chk.rows_cap, chk.status, kSiteDispatch)) continue;
        uint4* dst = reinterpret_cast<uint4*>(xq + row * H + b * 32);
        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        if ((b & 3) == 0) {
            const int rank = static_cast<int>(row) - off[p];
            *reinterpret_cast<uint32_t*>(xs_t + act_sf_offset(toff[p] + rank / tile, rank % tile, b, kchunks)) = sword;
        }
    }
}

// out[t][8c .. 8c+8) = bf16( sum_j w[t,j] * y[pos[t,j]][...] ), fp32, j in order.
// All k row loads are issued before the sum starts, so one thread keeps k
// 16-byte reads in flight instead of one.
__device__ __forceinline__ void combine_chunk(const __nv_bfloat16* __restrict__ y, const float* __restrict__ w,
                                              const int32_t* __restrict__ pos, int64_t t, int c, int H, int k,
                                              __nv_bfloat16* __restrict__ out, const DispatchBounds& chk)
{
    (void)chk;
    float wj[MM_MAX_TOPK];
    uint4 u[MM_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MM_MAX_TOPK; ++j) {
        if (j < k) {
            wj[j] = w[t * k + j];
            const int64_t row = pos[t * k + j];
            if (MM_CHECK(row >= 0 && row < chk.rows_cap, chk.status, kSiteCombine))
                u[j] = *(reinterpret_cast<const uint4*>(y + row * H) + c);
            else
                u[j] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < MM_MAX_TOPK; ++j) {
        if (j < k) {
            const uint32_t w4[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = fmaf(wj[j], __uint_as_float(w4[i] << 16), acc[2 * i]);
                acc[2 * i + 1] = fmaf(wj[j], __uint_as_float(w4[i] & 0xFFFF0000u), acc[2 * i + 1]);
            }
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    reinterpret_cast<uint4*>(out + t * H)[c] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace mm
