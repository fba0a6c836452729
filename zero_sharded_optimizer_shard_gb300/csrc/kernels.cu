// Streaming kernels of the ZeRO-3 step (sm_103a).
//
// Every kernel here is bound by HBM bandwidth: per element the fused step
// reads N_d bf16 gradients and the fp32 master/m/v and writes master/m/v,
// the bf16 shard and the bf16 all-gather copy, with about 20 binary32
// operations in between.  There is no contraction, so no tensor core work.
//
// Work layout.  A launch covers up to ZERO3_MAX_RANKS + 1 "spans"; a span is
// one owner's slice [lo, hi) of local indices (a rank's shard, or the
// persistent group, which the fused step takes as one more span when its
// gradients sit at one common offset from every rank's flat gradients).  The spans' elements are cut into chunks of 8 consecutive local
// indices aligned to multiples of 8, numbered consecutively across spans.
// Thread c of the grid takes chunk c, so the 32 lanes of a warp
// touch 32 adjacent chunks: 512 contiguous bytes of every bf16 stream and
// 1 KiB of every fp32 stream per warp instruction pair.  Interior chunks of a
// span use 16-byte accesses for the states and shards.  The gradient and
// all-gather streams start at r*S - origin and r*S, which need not be
// multiples of 8 elements: a chunk at a nonzero element phase reads the two
// aligned 16-byte blocks around it and realigns them (ld8_window), a whole
// warp of such chunks stores its all-gather values as aligned blocks passed
// between neighbouring lanes (st8_warp), chunks next to a span edge use the
// widest aligned width their phase allows, and the edge chunks themselves
// take the element-by-element path.
//
// Arithmetic per element follows the fixed order of the AdamW reading with
// IEEE round-to-nearest intrinsics (no contraction into FMA):
//   g = (sum_q f32(grad_q)) * inv_nd            (q ascending, from +0)
//   p = p*decay; m = b1*m + omb1*g; v = b2*v + omb2*(g*g)
//   d = sqrt(v)*inv_sqrt_bc2 + eps; p = p - step_size*(m/d); sparam = bf16(p)
#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "internal.h"

namespace z3 {

// Kernel parameters are passed by value; 32764 bytes is the limit.
static_assert(sizeof(StreamArgs) <= 32764, "StreamArgs exceeds the kernel parameter limit");

namespace {

__device__ __forceinline__ void adamw(float g, float& p, float& m, float& v, const Scalars& s) {
    p = __fmul_rn(p, s.decay);
    m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    const float d = __fadd_rn(__fmul_rn(__fsqrt_rn(v), s.inv_sqrt_bc2), s.eps);
    p = __fsub_rn(p, __fmul_rn(s.step_size, __fdiv_rn(m, d)));
}

// Streaming fp32 vector accesses of the optimizer states.
__device__ __forceinline__ float4 ldcs_f4(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void stcs_f4(float* p, float4 x) {
    __stcs(reinterpret_cast<float4*>(p), x);
}

// 8 consecutive bf16 values starting at an address of element phase ph
// (address / 2 mod 8): one 16-byte load when aligned, else the widest
// aligned loads (8, 4 or 2 bytes) through the read-only path, so that the
// bytes neighbouring threads share are served from L1.
__device__ __forceinline__ uint4 ld8_phase(const uint16_t* p, int ph) {
    if (ph == 0) return ldcs16(p);
    if ((ph & 3) == 0) {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
        const uint2 b = __ldg(reinterpret_cast<const uint2*>(p + 4));
        return make_uint4(a.x, a.y, b.x, b.y);
    }
    if ((ph & 1) == 0) {
        const unsigned int* q = reinterpret_cast<const unsigned int*>(p);
        return make_uint4(__ldg(q), __ldg(q + 1), __ldg(q + 2), __ldg(q + 3));
    }
    const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        w[k] = static_cast<uint32_t>(__ldg(q + 2 * k)) |
               (static_cast<uint32_t>(__ldg(q + 2 * k + 1)) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The 8 bf16 values at elements ph..ph+7 (1 <= ph <= 7) of the 16-element
// window formed by two consecutive aligned 16-byte blocks b0, b1 (window
// words w0..w7).  Branch-free, so the compiler keeps every rank's loads
// ahead of the first realignment: result word m is the funnel shift of
// words k+m and k+m+1 (k = ph / 2) right by 16 * (ph & 1) bits, the words
// picked by two rounds of selects (by 2 words, then by 1).
__device__ __forceinline__ uint4 realign8(const uint4& b0, const uint4& b1, int ph) {
    const bool by2 = (ph & 4) != 0, by1 = (ph & 2) != 0;
    const uint32_t sh = static_cast<uint32_t>(ph & 1) * 16u;
    const uint32_t t0 = by2 ? b0.z : b0.x, t1 = by2 ? b0.w : b0.y, t2 = by2 ? b1.x : b0.z;
    const uint32_t t3 = by2 ? b1.y : b0.w, t4 = by2 ? b1.z : b1.x, t5 = by2 ? b1.w : b1.y;
    const uint32_t v0 = by1 ? t1 : t0, v1 = by1 ? t2 : t1, v2 = by1 ? t3 : t2;
    const uint32_t v3 = by1 ? t4 : t3, v4 = by1 ? t5 : t4;
    return make_uint4(__funnelshift_r(v0, v1, sh), __funnelshift_r(v1, v2, sh),
                      __funnelshift_r(v2, v3, sh), __funnelshift_r(v3, v4, sh));
}

// 8 consecutive bf16 values at p, element phase ph != 0, read as the two
// aligned 16-byte blocks around them (through the read-only path, so the
// block a neighbouring thread also reads is served from L1).  The caller
// guarantees that both blocks lie inside the valid range: the 8 elements
// before p and the 16 from p on.
__device__ __forceinline__ uint4 ld8_window(const uint16_t* p, int ph) {
    const uint16_t* a = p - ph;
    const uint4 b0 = __ldg(reinterpret_cast<const uint4*>(a));
    const uint4 b1 = __ldg(reinterpret_cast<const uint4*>(a + 8));
    return realign8(b0, b1, ph);
}

// 8 consecutive bf16 values stored at an address of element phase ph.
__device__ __forceinline__ void st8_phase(uint16_t* p, int ph, const uint4& h) {
    if (ph == 0) {
        stcs16(p, h);
    } else if ((ph & 3) == 0) {
        __stcs(reinterpret_cast<uint2*>(p), make_uint2(h.x, h.y));
        __stcs(reinterpret_cast<uint2*>(p + 4), make_uint2(h.z, h.w));
    } else if ((ph & 1) == 0) {
        unsigned int* q = reinterpret_cast<unsigned int*>(p);
        __stcs(q, h.x);
        __stcs(q + 1, h.y);
        __stcs(q + 2, h.z);
        __stcs(q + 3, h.w);
    } else {
        const uint32_t w[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            p[2 * k] = static_cast<uint16_t>(w[k] & 0xffffu);
            p[2 * k + 1] = static_cast<uint16_t>(w[k] >> 16);
        }
    }
}

// Warp-cooperative store of a phased stream (1 <= ph <= 7).  All 32 lanes of
// the warp hold consecutive chunks of one span, so lane i's 8 values go to
// p + 8 i.  The aligned 16-byte block starting at lane i's element 8 - ph
// holds lane i's last ph values and lane i+1's first 8 - ph: lanes 0..30
// store that block (warp_block builds it, the neighbour's values coming by
// shuffle), lane 31 stores its last ph values and lane 0 its first 8 - ph
// values element by element.  Every element of the warp's range is written
// exactly once and nothing outside it.  Every lane of the warp must call
// warp_block.
__device__ __forceinline__ uint4 warp_block(int ph, const uint4& h) {
    uint4 n;
    n.x = __shfl_down_sync(0xffffffffu, h.x, 1);
    n.y = __shfl_down_sync(0xffffffffu, h.y, 1);
    n.z = __shfl_down_sync(0xffffffffu, h.z, 1);
    n.w = __shfl_down_sync(0xffffffffu, h.w, 1);
    return realign8(h, n, 8 - ph);
}

__device__ __forceinline__ void st8_warp(uint16_t* p, int ph, const uint4& h, const uint4& blk) {
    const int lane = threadIdx.x & 31;
    const int k = 8 - ph;
    if (lane < 31) stcs16(p + k, blk);
    if (lane == 0 || lane == 31) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t w = e < 2 ? h.x : (e < 4 ? h.y : (e < 6 ? h.z : h.w));
            const uint16_t v = static_cast<uint16_t>((e & 1) ? (w >> 16) : (w & 0xffffu));
            if (lane == 0 ? e < k : e >= k) p[e] = v;
        }
    }
}

// Reduced gradient of 8 consecutive elements, ranks summed in ascending
// order; ph is the element phase of the gradient streams (equal for every
// rank).  `window`: the chunk's neighbours on both sides lie in the span, so
// a phased chunk may be read as the two aligned 16-byte blocks around it.
// All loads are issued before the first add.
template <int ND>
__device__ __forceinline__ void reduce8(const StreamArgs& a, int64_t off, int ph, bool window,
                                        float* g) {
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = 0.0f;
    if constexpr (ND > 0) {
        uint4 raw[ND];
        if (ph == 0) {
#pragma unroll
            for (int q = 0; q < ND; ++q) raw[q] = ldcs16(a.grads[q] + off);
        } else if (window) {
#pragma unroll
            for (int q = 0; q < ND; ++q) raw[q] = ld8_window(a.grads[q] + off, ph);
        } else {
#pragma unroll
            for (int q = 0; q < ND; ++q) raw[q] = ld8_phase(a.grads[q] + off, ph);
        }
#pragma unroll
        for (int q = 0; q < ND; ++q) {
            float f[8];
            unpack8(raw[q], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) g[e] = __fadd_rn(g[e], f[e]);
        }
    } else {
        const int nd = a.nd;
        for (int q0 = 0; q0 < nd; q0 += 8) {
            uint4 raw[8];
            const int n = (nd - q0) < 8 ? (nd - q0) : 8;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < n) raw[k] = ld8_phase(a.grads[q0 + k] + off, ph);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (k < n) {
                    float f[8];
                    unpack8(raw[k], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) g[e] = __fadd_rn(g[e], f[e]);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = __fmul_rn(g[e], a.sc.inv_nd);
}

template <int ND>
__device__ __forceinline__ float reduce1(const StreamArgs& a, int64_t off) {
    float s = 0.0f;
    const int nd = ND > 0 ? ND : a.nd;
    for (int q = 0; q < nd; ++q) s = __fadd_rn(s, bf16_f32(a.grads[q][off]));
    return __fmul_rn(s, a.sc.inv_nd);
}

template <int MODE, int ND, int GT>
__device__ __forceinline__ void vector_chunk(const StreamArgs& a, const Span& sp, int64_t i0,
                                             float* hq, bool warp_store) {
    float g[8];
    if constexpr (MODE == kFused || MODE == kFusedRep || MODE == kFusedQ || MODE == kReduce) {
        // blocks of a phased chunk: local [i0 - ph, i0 - ph + 16) within [i0 - 8, i0 + 16)
        const bool window = i0 - 8 >= sp.lo && i0 + 16 <= sp.hi;
        reduce8<ND>(a, sp.gofs + i0, sp.gphase, window, g);
    }
    if constexpr (MODE == kQuant) {
        unpack8(ldcs16(static_cast<const uint16_t*>(sp.in) + i0), hq);
        return;
    }
    if constexpr (MODE == kReduce) {
        if constexpr (GT == ZERO3_BF16) {
            stcs16(static_cast<uint16_t*>(sp.out) + i0, pack8(g));
        } else {
            float* o = static_cast<float*>(sp.out) + i0;
            stcs_f4(o, make_float4(g[0], g[1], g[2], g[3]));
            stcs_f4(o + 4, make_float4(g[4], g[5], g[6], g[7]));
        }
        return;
    }
    if constexpr (MODE == kAdam) {
        if constexpr (GT == ZERO3_BF16) {
            unpack8(ldcs16(static_cast<const uint16_t*>(sp.in) + i0), g);
        } else {
            const float* in = static_cast<const float*>(sp.in) + i0;
            const float4 g0 = ldcs_f4(in), g1 = ldcs_f4(in + 4);
            g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
            g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
        }
    }
    float p[8];
    if constexpr (MODE == kCast) {
        const float* in = static_cast<const float*>(sp.in) + i0;
        const float4 p0 = ldcs_f4(in), p1 = ldcs_f4(in + 4);
        p[0] = p0.x; p[1] = p0.y; p[2] = p0.z; p[3] = p0.w;
        p[4] = p1.x; p[5] = p1.y; p[6] = p1.z; p[7] = p1.w;
    } else {
        float m[8], v[8];
        const float4 p0 = ldcs_f4(sp.master + i0), p1 = ldcs_f4(sp.master + i0 + 4);
        const float4 m0 = ldcs_f4(sp.m + i0), m1 = ldcs_f4(sp.m + i0 + 4);
        const float4 v0 = ldcs_f4(sp.v + i0), v1 = ldcs_f4(sp.v + i0 + 4);
        p[0] = p0.x; p[1] = p0.y; p[2] = p0.z; p[3] = p0.w;
        p[4] = p1.x; p[5] = p1.y; p[6] = p1.z; p[7] = p1.w;
        m[0] = m0.x; m[1] = m0.y; m[2] = m0.z; m[3] = m0.w;
        m[4] = m1.x; m[5] = m1.y; m[6] = m1.z; m[7] = m1.w;
        v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
        v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
#pragma unroll
        for (int e = 0; e < 8; ++e) adamw(g[e], p[e], m[e], v[e], a.sc);
        stcs_f4(sp.master + i0, make_float4(p[0], p[1], p[2], p[3]));
        stcs_f4(sp.master + i0 + 4, make_float4(p[4], p[5], p[6], p[7]));
        stcs_f4(sp.m + i0, make_float4(m[0], m[1], m[2], m[3]));
        stcs_f4(sp.m + i0 + 4, make_float4(m[4], m[5], m[6], m[7]));
        stcs_f4(sp.v + i0, make_float4(v[0], v[1], v[2], v[3]));
        stcs_f4(sp.v + i0 + 4, make_float4(v[4], v[5], v[6], v[7]));
    }
    const uint4 h = pack8(p);
    if constexpr (MODE == kFusedQ) unpack8(h, hq);
    uint4 blk = h;
    if (warp_store) blk = warp_block(sp.fphase, h);
    if constexpr (MODE == kFusedRep) {
        // all-gather into every rank's full parameter copy
        const int nd = ND > 0 ? ND : a.nd;
#pragma unroll
        for (int q = 0; q < (ND > 0 ? ND : ZERO3_MAX_RANKS); ++q) {
            if (ND == 0 && q >= nd) break;
            if (warp_store)
                st8_warp(a.reps[q] + sp.fofs + i0, sp.fphase, h, blk);
            else
                st8_phase(a.reps[q] + sp.fofs + i0, sp.fphase, h);
        }
    } else {
        stcs16(static_cast<uint16_t*>(sp.out) + i0, h);
        if (warp_store)
            st8_warp(a.full + sp.fofs + i0, sp.fphase, h, blk);
        else if (sp.fofs >= 0)
            st8_phase(a.full + sp.fofs + i0, sp.fphase, h);
    }
}

template <int MODE, int ND, int GT>
__device__ __forceinline__ void scalar_chunk(const StreamArgs& a, const Span& sp, int64_t i0,
                                             float* hq) {
    for (int e = 0; e < 8; ++e) {
        const int64_t i = i0 + e;
        if constexpr (MODE == kFusedQ || MODE == kQuant) hq[e] = 0.0f;
        if (i < sp.lo || i >= sp.hi) continue;
        if constexpr (MODE == kQuant) {
            hq[e] = bf16_f32(static_cast<const uint16_t*>(sp.in)[i]);
            continue;
        }
        float g = 0.0f;
        if constexpr (MODE == kFused || MODE == kFusedRep || MODE == kFusedQ || MODE == kReduce)
            g = reduce1<ND>(a, sp.gofs + i);
        if constexpr (MODE == kReduce) {
            if constexpr (GT == ZERO3_BF16)
                static_cast<uint16_t*>(sp.out)[i] = to_bf16(g);
            else
                static_cast<float*>(sp.out)[i] = g;
            continue;
        }
        if constexpr (MODE == kAdam) {
            if constexpr (GT == ZERO3_BF16)
                g = bf16_f32(static_cast<const uint16_t*>(sp.in)[i]);
            else
                g = static_cast<const float*>(sp.in)[i];
        }
        float p;
        if constexpr (MODE == kCast) {
            p = static_cast<const float*>(sp.in)[i];
        } else {
            p = sp.master[i];
            float m = sp.m[i], v = sp.v[i];
            adamw(g, p, m, v, a.sc);
            sp.master[i] = p;
            sp.m[i] = m;
            sp.v[i] = v;
        }
        const uint16_t h = to_bf16(p);
        if constexpr (MODE == kFusedQ) hq[e] = bf16_f32(h);
        if constexpr (MODE == kFusedRep) {
            const int nd = ND > 0 ? ND : a.nd;
            for (int q = 0; q < nd; ++q) a.reps[q][sp.fofs + i] = h;
        } else {
            static_cast<uint16_t*>(sp.out)[i] = h;
            if (sp.fofs >= 0) a.full[sp.fofs + i] = h;
        }
    }
}

// qwZ epilogue: the warp's 32 chunks are one 256-element block of one shard
// (the launch numbers chunks that way).  absmax by warp shuffle, then with
// qmax = 2^(BITS-1) - 1: scale = absmax/qmax, code = round-half-even(x *
// qmax/absmax), one binary32 operation each.  int8 codes take a byte each;
// int4 codes two per byte, element 2j in the low nibble.  Every lane of the
// warp reaches the shuffles.
template <int BITS>
__device__ __forceinline__ void qwz_block(const Span& sp, int64_t i0, const float* hq) {
    constexpr float kQmax = BITS == 4 ? 7.0f : 127.0f;
    constexpr int kQi = BITS == 4 ? 7 : 127;
    float am = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(hq[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const float inv = am > 0.0f ? __fdiv_rn(kQmax, am) : 0.0f;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        int q = __float2int_rn(__fmul_rn(hq[e], inv));
        q = q > kQi ? kQi : (q < -kQi ? -kQi : q);
        if constexpr (BITS == 4)
            w[0] |= (static_cast<uint32_t>(q) & 0xfu) << (4 * e);
        else
            w[e >> 2] |= (static_cast<uint32_t>(q) & 0xffu) << (8 * (e & 3));
    }
    if (i0 >= sp.hi) return;  // chunk past the shard's end: nothing to store
    if ((threadIdx.x & 31) == 0) sp.scales[i0 / kQwzBlock] = __fdiv_rn(am, kQmax);
    uint8_t* bytes = reinterpret_cast<uint8_t*>(sp.codes);
    if constexpr (BITS == 4) {
        if (i0 + 8 <= sp.hi) {
            *reinterpret_cast<uint32_t*>(bytes + i0 / 2) = w[0];
        } else {  // shard end: ceil((hi - i0) / 2) bytes, unused nibbles are 0
            for (int b = 0; 2 * b < sp.hi - i0; ++b)
                bytes[i0 / 2 + b] = static_cast<uint8_t>((w[0] >> (8 * b)) & 0xffu);
        }
    } else {
        if (i0 + 8 <= sp.hi) {
            *reinterpret_cast<uint2*>(bytes + i0) = make_uint2(w[0], w[1]);
        } else {
            for (int e = 0; e < 8 && i0 + e < sp.hi; ++e)
                bytes[i0 + e] = static_cast<uint8_t>((w[e >> 2] >> (8 * (e & 3))) & 0xffu);
        }
    }
}

// Resident blocks of 256 threads per SM that the register allocation must
// allow.  The modes that reduce gradients with a compile-time rank count keep
// 4 (at most 64 registers a thread): the ZeRO-1/2 step at N_d = 8 otherwise
// takes 75 and the reduce-scatter 80, and both drop to 3 blocks.  None of
// them spills.
template <int MODE, int ND>
__host__ __device__ constexpr int min_blocks_per_sm() {
    return (ND > 0 && (MODE == kFused || MODE == kFusedRep || MODE == kFusedQ ||
                       MODE == kReduce))
               ? 4
               : 1;
}

template <int MODE, int ND, int GT>
__global__ void __launch_bounds__(kThreads, min_blocks_per_sm<MODE, ND>())
    stream_kernel(const __grid_constant__ StreamArgs a) {
    wait_prior_grids();
    allow_next_grid();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int s = 0;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         base < a.total_chunks; base += stride) {
        // one chunk per thread (the single-iteration loop keeps the code
        // shape under which no instantiation spills)
#pragma unroll
        for (int j = 0; j < 1; ++j) {
            const int64_t c = base + static_cast<int64_t>(j) * blockDim.x;
            if (c >= a.total_chunks) break;
            while (s + 1 < a.n_spans && c >= a.span[s + 1].chunk0) ++s;
            const Span& sp = a.span[s];
            const int64_t i0 = (sp.lo & ~static_cast<int64_t>(7)) + ((c - sp.chunk0) << 3);
            float hq[8];
            const bool vec = i0 >= sp.lo && i0 + 8 <= sp.hi;
            // A phased all-gather stream is stored by the whole warp at once
            // when its 32 lanes hold vector chunks of one span (a
            // warp-uniform decision: every active lane takes part in it, and
            // a partial or diverged warp keeps the per-lane stores).
            bool warp_store = false;
            if constexpr (MODE == kFused || MODE == kFusedRep || MODE == kFusedQ) {
                const unsigned active = __activemask();
                if (active == 0xffffffffu) {
                    const int s0 = __shfl_sync(0xffffffffu, s, 0);
                    warp_store = __all_sync(0xffffffffu, vec && s == s0 && sp.fofs >= 0 &&
                                                             sp.fphase != 0);
                }
            }
            if (vec)
                vector_chunk<MODE, ND, GT>(a, sp, i0, hq, warp_store);
            else
                scalar_chunk<MODE, ND, GT>(a, sp, i0, hq);
            if constexpr (MODE == kFusedQ || MODE == kQuant)
                qwz_block<GT == 4 ? 4 : 8>(sp, i0, hq);
        }
    }
}

// The grid covers every chunk once (the grid-stride loop in the kernels only
// matters beyond 2^31-1 blocks).
// Measured on GB300 at 1.3B / N_d = 8 this keeps more independent requests
// in flight than an SM-sized persistent grid, whose threads serialise
// load -> compute -> store per iteration: 7.2 TB/s against 6.5 TB/s.
int grid_for(int64_t total_chunks, int chunks_per_thread = 1) {
    const int64_t per = static_cast<int64_t>(kThreads) * chunks_per_thread;
    const int64_t need = (total_chunks + per - 1) / per;
    const int64_t cap = 0x7fffffff;
    return static_cast<int>(need < cap ? need : cap);
}

template <int MODE, int ND, int GT>
cudaError_t launch_one(const StreamArgs& a, cudaStream_t stream) {
    const int grid = grid_for(a.total_chunks);
    if (grid <= 0) return cudaSuccess;
    const cudaError_t e = launch_programmatic(stream_kernel<MODE, ND, GT>, grid, a, stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int MODE, int GT>
cudaError_t launch_nd(const StreamArgs& a, cudaStream_t stream) {
    switch (a.nd) {
        case 1: return launch_one<MODE, 1, GT>(a, stream);
        case 2: return launch_one<MODE, 2, GT>(a, stream);
        case 3: return launch_one<MODE, 3, GT>(a, stream);
        case 4: return launch_one<MODE, 4, GT>(a, stream);
        case 5: return launch_one<MODE, 5, GT>(a, stream);
        case 6: return launch_one<MODE, 6, GT>(a, stream);
        case 7: return launch_one<MODE, 7, GT>(a, stream);
        case 8: return launch_one<MODE, 8, GT>(a, stream);
        default: return launch_one<MODE, 0, GT>(a, stream);
    }
}

}  // namespace

cudaError_t launch_stream(int mode, const StreamArgs& a, cudaStream_t stream) {
    if (a.total_chunks <= 0) return cudaSuccess;
    switch (mode) {
        case kFused: return launch_nd<kFused, 0>(a, stream);
        case kFusedRep: return launch_nd<kFusedRep, 0>(a, stream);
        // qwZ modes: the template's GT carries the code width (8 or 4 bits)
        case kFusedQ:
            return a.dtype == 4 ? launch_nd<kFusedQ, 4>(a, stream) : launch_nd<kFusedQ, 8>(a, stream);
        case kQuant:
            return a.dtype == 4 ? launch_one<kQuant, 1, 4>(a, stream)
                                : launch_one<kQuant, 1, 8>(a, stream);
        case kReduce:
            return a.dtype == ZERO3_BF16 ? launch_nd<kReduce, ZERO3_BF16>(a, stream)
                                         : launch_nd<kReduce, ZERO3_F32>(a, stream);
        case kAdam:
            return a.dtype == ZERO3_BF16 ? launch_one<kAdam, 1, ZERO3_BF16>(a, stream)
                                         : launch_one<kAdam, 1, ZERO3_F32>(a, stream);
        case kCast: return launch_one<kCast, 1, 0>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace z3
