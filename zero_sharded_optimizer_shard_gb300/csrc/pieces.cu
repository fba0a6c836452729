// The piece kernel of the copy-like launches (sm_103a): submodule gathers
// (one or several submodules per launch), the all-gather copy of the shards
// into the flat parameter buffer, and the dequantizing qwZ all-gather.
#include <cuda_runtime.h>

#include <cstdint>

#include "device_common.cuh"
#include "internal.h"

namespace z3 {

// Kernel parameters are passed by value; 32764 bytes is the limit.
static_assert(sizeof(PieceArgs<kLargePieces>) <= 32764, "PieceArgs exceeds the kernel parameter limit");

namespace {

// Copy-like work: submodule gathers (one or many submodules per launch), the
// all-gather copy sparam -> full and the dequantizing qwZ all-gather.  Every
// byte moves once, so the kernel is bound by HBM bandwidth with few
// operations per byte; what matters is many independent 16-byte requests in
// flight and no narrow or partial accesses.
//
// Chunks are aligned to the DESTINATION, so every store is one aligned
// 16-byte store; a source at a nonzero phase is realigned on the way in.
// A warp's 32 lanes hold 32 consecutive chunks of one piece (per step j of
// the thread's four chunks), so lane l loads the aligned source unit under
// its chunk and takes lane l+1's by shuffle (lane 31 loads the one after):
// one aligned load per chunk.  Chunks whose source units would reach past
// either end of the piece (at most two per piece edge) are copied element by
// element.  Each lane issues all of its loads before its first store (the
// compiler cannot move a load above a store through a possibly aliasing
// pointer, which would leave one load in flight per lane).
constexpr int kPieceChunks = kPieceWarpChunks / 32;   // chunks per lane

// Source unit of a chunk and its realignment, per kind.
//   bf16: 8 elements per aligned 16-byte unit; PH elements.
//   int8: 8 codes per aligned 8-byte unit; PH bytes.
//   int4: 8 codes per aligned 4-byte unit; PH nibbles.
// The phase is the same for a whole piece, hence for a whole warp, so the
// realignment is compiled per phase: a few funnel shifts of fixed words.
template <int KIND>
struct Unit;
template <>
struct Unit<kPieceBf16> {
    using T = uint4;
    static constexpr int kUnitBytes = 16;  // bytes of 8 source elements
    static __device__ __forceinline__ const char* at(const void* src, int64_t idx) {
        return static_cast<const char*>(src) + idx * 2;
    }
    static __device__ __forceinline__ T load(const char* p) { return ldcs16(p); }
    static __device__ __forceinline__ T shfl(const T& x) {
        T n;
        n.x = __shfl_down_sync(0xffffffffu, x.x, 1);
        n.y = __shfl_down_sync(0xffffffffu, x.y, 1);
        n.z = __shfl_down_sync(0xffffffffu, x.z, 1);
        n.w = __shfl_down_sync(0xffffffffu, x.w, 1);
        return n;
    }
    // elements PH..PH+7 of the 16 elements a, b: words k..k+4 (k = PH / 2)
    // funnel-shifted right by 16 * (PH % 2) bits
    template <int PH>
    static __device__ __forceinline__ T realign(const T& a, const T& b) {
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        constexpr int k = PH / 2;
        constexpr uint32_t sh = (PH & 1) * 16u;
        if constexpr (sh == 0) return make_uint4(w[k], w[k + 1], w[k + 2], w[k + 3]);
        return make_uint4(__funnelshift_r(w[k], w[k + 1], sh), __funnelshift_r(w[k + 1], w[k + 2], sh),
                          __funnelshift_r(w[k + 2], w[k + 3], sh),
                          __funnelshift_r(w[k + 3], w[k + 4], sh));
    }
};
template <>
struct Unit<kPieceInt8> {
    using T = uint2;
    static constexpr int kUnitBytes = 8;
    static __device__ __forceinline__ const char* at(const void* src, int64_t idx) {
        return static_cast<const char*>(src) + idx;
    }
    static __device__ __forceinline__ T load(const char* p) {
        return __ldcs(reinterpret_cast<const uint2*>(p));
    }
    static __device__ __forceinline__ T shfl(const T& x) {
        return make_uint2(__shfl_down_sync(0xffffffffu, x.x, 1),
                          __shfl_down_sync(0xffffffffu, x.y, 1));
    }
    // bytes PH..PH+7 of the 16 bytes a, b
    template <int PH>
    static __device__ __forceinline__ T realign(const T& a, const T& b) {
        const uint32_t w[4] = {a.x, a.y, b.x, b.y};
        constexpr int k = PH / 4;
        constexpr uint32_t sh = (PH & 3) * 8u;
        if constexpr (sh == 0) return make_uint2(w[k], w[k + 1]);
        return make_uint2(__funnelshift_r(w[k], w[k + 1], sh), __funnelshift_r(w[k + 1], w[k + 2], sh));
    }
};
template <>
struct Unit<kPieceInt4> {
    using T = uint32_t;
    static constexpr int kUnitBytes = 4;
    // idx is a multiple of 8 wherever a unit is read (an aligned unit)
    static __device__ __forceinline__ const char* at(const void* src, int64_t idx) {
        return static_cast<const char*>(src) + idx / 2;
    }
    static __device__ __forceinline__ T load(const char* p) {
        return __ldcs(reinterpret_cast<const unsigned int*>(p));
    }
    static __device__ __forceinline__ T shfl(const T& x) {
        return __shfl_down_sync(0xffffffffu, x, 1);
    }
    template <int PH>
    static __device__ __forceinline__ T realign(const T& a, const T& b) {
        return __funnelshift_r(a, b, PH * 4u);
    }
};

// Exact binary32 value of a code without a conversion instruction: the code
// plus a bias (128 for int8, 8 for int4) is an integer below 2^8, placed in
// the low mantissa bits of 2^23; subtracting 2^23 + bias is exact.
__device__ __forceinline__ float int8_code_f32(uint32_t biased_word, int k) {
    // byte k of the biased word under the exponent byte 0x4B (2^23)
    const uint32_t v = __byte_perm(biased_word, 0x4B000000u, 0x7650u | static_cast<uint32_t>(k));
    return __fsub_rn(__uint_as_float(v), 8388736.0f);  // 2^23 + 128
}
// int4: the biased nibbles split once into two words of one nibble per byte
// (even codes from the low nibbles, odd codes from the high ones), then the
// same byte permute as int8.
__device__ __forceinline__ float int4_code_f32(uint32_t nibble_bytes, int k) {
    const uint32_t v = __byte_perm(nibble_bytes, 0x4B000000u, 0x7650u | static_cast<uint32_t>(k));
    return __fsub_rn(__uint_as_float(v), 8388616.0f);  // 2^23 + 8
}

// The 8 codes of a realigned unit as binary32.
template <int KIND>
__device__ __forceinline__ void codes_f32(const typename Unit<KIND>::T& u, float* f) {
    if constexpr (KIND == kPieceInt4) {
        const uint32_t x = u ^ 0x88888888u;
        const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = int4_code_f32((e & 1) ? hi : lo, e >> 1);
    } else {
        const uint32_t x0 = u.x ^ 0x80808080u, x1 = u.y ^ 0x80808080u;
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = int8_code_f32(e < 4 ? x0 : x1, e & 3);
    }
}

// Destination element d of piece P, element by element (chunks at the
// piece's edges).
template <int KIND>
__device__ __forceinline__ uint16_t piece_element(const Piece& P, int64_t d) {
    const int64_t e = P.s0 + d;
    if constexpr (KIND == kPieceBf16) {
        return static_cast<const uint16_t*>(P.src)[e];
    } else {
        int c;
        if constexpr (KIND == kPieceInt4) {
            const uint32_t b = static_cast<const uint8_t*>(P.src)[e / 2];
            c = static_cast<int>(b << (28 - 4 * (e & 1))) >> 28;
        } else {
            c = static_cast<const int8_t*>(P.src)[e];
        }
        return to_bf16(__fmul_rn(static_cast<float>(c), P.scales[e / kQwzBlock]));
    }
}

// Phase 2 of a warp's chunks at source phase PH: take the neighbour's unit
// by shuffle (lane 31 loaded its own), realign, convert and store the vector
// chunks.  Every lane of the warp calls this (the shuffles need all of
// them).
// Dequantizing kinds: y = bf16_rne(f32(code) * scale), with each element's
// own 256-element block scale; only a chunk whose source starts in the last
// 7 elements of a block (possible when PH != 0) straddles two blocks, and its
// tail takes the second scale (a select per element: measured cheaper than a
// fix-up branch, which the compiler predicates).
template <int KIND, int PH>
__device__ __forceinline__ void piece_phase2(uint16_t* dst, int64_t x0, int lane,
                                             typename Unit<KIND>::T* cur,
                                             const typename Unit<KIND>::T* nxt, const bool* vec,
                                             const float* sc0, const float* sc1) {
    using U = Unit<KIND>;
    // elements of a chunk in its first block: all 8 unless a phased chunk's
    // source starts in the block's last 7 elements (the same for the lane's
    // four chunks, which lie 256 elements apart)
    int split = 8;
    if constexpr (PH != 0 && KIND != kPieceBf16) {
        const uint32_t in_block = static_cast<uint32_t>(x0) % kQwzBlock;  // x0 >= 0
        if (in_block > kQwzBlock - 8) split = static_cast<int>(kQwzBlock - in_block);
    }
#pragma unroll
    for (int j = 0; j < kPieceChunks; ++j) {
        typename U::T u = cur[j];
        if constexpr (PH != 0) {
            const typename U::T n = U::shfl(cur[j]);
            u = U::template realign<PH>(cur[j], lane == 31 ? nxt[j] : n);
        }
        if (!vec[j]) continue;
        uint4 x;
        if constexpr (KIND == kPieceBf16) {
            x = u;
        } else {
            float y[8];
            codes_f32<KIND>(u, y);
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(y[e], e < split ? sc0[j] : sc1[j]);
            x = pack8(y);
        }
        // plain stores: evict-first stores measured slower for the
        // dequantizing all-gather (0.71 against 0.66 ms at 1.3B)
        *reinterpret_cast<uint4*>(dst + 256 * j) = x;
    }
}

// PHASED: some piece of the launch has a nonzero source phase; the aligned
// instantiation has no shuffles and fewer registers.
template <int KIND, bool PHASED, int MAXP>
__global__ void __launch_bounds__(kThreads, PHASED ? 4 : 5)
    piece_kernel(const __grid_constant__ PieceArgs<MAXP> a) {
    wait_prior_grids();
    allow_next_grid();
    using U = Unit<KIND>;
    const uint32_t w = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (w >= a.warp0[a.n]) return;  // whole warps leave together
    // the piece of warp w: the last i with warp0[i] <= w (same for every lane)
    int lo = 0, hi = a.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.warp0[mid] <= w)
            lo = mid;
        else
            hi = mid - 1;
    }
    const Piece& P = a.piece[lo];
    const int lane = threadIdx.x & 31;
    const int ph = PHASED ? P.ph : 0;
    // destination index of the warp's first element, and of the lane's chunk
    // at step 0 (step j adds 256: 32 lanes of 8 elements)
    const int64_t wbase = static_cast<int64_t>(w - a.warp0[lo]) * (kPieceWarpChunks * 8);
    const int64_t d00 = wbase + 8 * lane;
    const int64_t x0 = P.s0 + d00;  // its source index
    const char* src = U::at(P.src, x0 - ph);  // the aligned source unit under it
    constexpr int kStep = 32 * U::kUnitBytes;
    typename U::T cur[kPieceChunks], nxt[kPieceChunks];
    bool vec[kPieceChunks];
    float sc0[kPieceChunks], sc1[kPieceChunks];
    // Phase 1: every load of the vector chunks (codes or values, block
    // scales).  A warp whose 1024 elements and the units around them lie
    // inside the piece (nearly all warps) needs no per-chunk bounds.
    const bool interior = wbase >= P.lo + 8 && wbase + kPieceWarpChunks * 8 + 8 <= P.hi;
    if (interior) {
#pragma unroll
        for (int j = 0; j < kPieceChunks; ++j) {
            vec[j] = true;
            cur[j] = U::load(src + j * kStep);
            if (PHASED && ph && lane == 31) nxt[j] = U::load(src + j * kStep + U::kUnitBytes);
        }
    } else {
#pragma unroll
        for (int j = 0; j < kPieceChunks; ++j) {
            // the source unit under the chunk starts at destination index b
            const int64_t b = d00 + 256 * j - ph;
            vec[j] = b >= P.lo && b + (ph ? 16 : 8) <= P.hi;
            if (b >= P.lo && b + 8 <= P.hi) cur[j] = U::load(src + j * kStep);
            if (PHASED && ph && lane == 31 && vec[j])
                nxt[j] = U::load(src + j * kStep + U::kUnitBytes);
        }
    }
    // Block scales of the vector chunks: the chunk's first element's block,
    // and its last element's (the same one unless a phased chunk straddles
    // two blocks).
    if constexpr (KIND != kPieceBf16) {
        if (interior) {
            // x0 >= 0: the warp starts past the piece's first element
            const float* s0p = P.scales + static_cast<uint64_t>(x0) / kQwzBlock;
            const float* s1p = P.scales + static_cast<uint64_t>(x0 + 7) / kQwzBlock;
#pragma unroll
            for (int j = 0; j < kPieceChunks; ++j) {
                sc0[j] = s0p[j];
                if constexpr (PHASED) sc1[j] = s1p[j];
            }
        } else {
            // x0 itself may lie before the piece (negative) on an edge lane;
            // a vector chunk's own source index x0 + 256 j never does
#pragma unroll
            for (int j = 0; j < kPieceChunks; ++j) {
                if (vec[j]) {
                    const uint64_t xj = static_cast<uint64_t>(x0 + 256 * j);
                    sc0[j] = P.scales[xj / kQwzBlock];
                    if constexpr (PHASED) sc1[j] = P.scales[(xj + 7) / kQwzBlock];
                }
            }
        }
    }
    uint16_t* dst = P.dst + d00;
    if constexpr (!PHASED) {
        piece_phase2<KIND, 0>(dst, x0, lane, cur, nxt, vec, sc0, sc1);
    } else {
        switch (ph) {  // warp-uniform
            case 0: piece_phase2<KIND, 0>(dst, x0, lane, cur, nxt, vec, sc0, sc1); break;
            case 1: piece_phase2<KIND, 1>(dst, x0, lane, cur, nxt, vec, sc0, sc1); break;
            case 2: piece_phase2<KIND, 2>(dst, x0, lane, cur, nxt, vec, sc0, sc1); break;
            case 3: piece_phase2<KIND, 3>(dst, x0, lane, cur, nxt, vec, sc0, sc1); break;
            case 4: piece_phase2<KIND, 4>(dst, x0, lane, cur, nxt, vec, sc0, sc1); break;
            case 5: piece_phase2<KIND, 5>(dst, x0, lane, cur, nxt, vec, sc0, sc1); break;
            case 6: piece_phase2<KIND, 6>(dst, x0, lane, cur, nxt, vec, sc0, sc1); break;
            default: piece_phase2<KIND, 7>(dst, x0, lane, cur, nxt, vec, sc0, sc1); break;
        }
    }
    // Phase 3: the chunks at the piece's edges, element by element.  Kept out
    // of the load phase: with its stores between the loads, the loads of the
    // later chunks were no longer all in flight together (measured: the int8
    // dequantizing all-gather at 1.3B took 0.84 ms instead of 0.66 ms).
    if (!interior) {
#pragma unroll
        for (int j = 0; j < kPieceChunks; ++j) {
            if (vec[j]) continue;
            const int64_t d0 = d00 + 256 * j;
            const int64_t e0 = d0 > P.lo ? d0 : P.lo;
            const int64_t e1 = d0 + 8 < P.hi ? d0 + 8 : P.hi;
            for (int64_t d = e0; d < e1; ++d) P.dst[d] = piece_element<KIND>(P, d);
        }
    }
}

template <int KIND, int MAXP>
cudaError_t launch_pieces(const PieceArgs<MAXP>& a, cudaStream_t stream) {
    const uint32_t warps = a.warp0[a.n];
    if (a.n <= 0 || warps == 0) return cudaSuccess;
    const int grid = static_cast<int>((warps + kThreads / 32 - 1) / (kThreads / 32));
    bool phased = false;
    for (int i = 0; i < a.n; ++i) phased = phased || a.piece[i].ph != 0;
    const cudaError_t e =
        phased ? launch_programmatic(piece_kernel<KIND, true, MAXP>, grid, a, stream)
               : launch_programmatic(piece_kernel<KIND, false, MAXP>, grid, a, stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int MAXP>
cudaError_t launch_pieces_kind(int kind, const PieceArgs<MAXP>& a, cudaStream_t stream) {
    switch (kind) {
        case kPieceBf16: return launch_pieces<kPieceBf16>(a, stream);
        case kPieceInt8: return launch_pieces<kPieceInt8>(a, stream);
        case kPieceInt4: return launch_pieces<kPieceInt4>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_pieces_small(int kind, const PieceArgs<kSmallPieces>& a, cudaStream_t stream) {
    return launch_pieces_kind(kind, a, stream);
}

cudaError_t launch_pieces_large(int kind, const PieceArgs<kLargePieces>& a, cudaStream_t stream) {
    return launch_pieces_kind(kind, a, stream);
}

}  // namespace z3
