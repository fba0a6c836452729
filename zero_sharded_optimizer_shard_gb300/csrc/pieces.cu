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
// 16-byte store; a source at a nonzero phase is realigned on the way.  A
// warp's 32 lanes hold 32 consecutive chunks of one piece per step j of the
// lane's chunks (four, or six in a phased dequantizing launch), so lane l
// loads the aligned source unit under its chunk and takes lane l+1's by
// shuffle: one aligned load per chunk.  The copy realigns the loaded units
// (lane 31 loads the unit after its own); a dequantizing warp first
// dequantizes every unit and realigns the bf16 results.  Chunks whose source
// units would reach past either end of the piece (at most two per piece
// edge) are copied element by element.  Each lane issues all of its loads
// before its first store (the compiler cannot move a load above a store
// through a possibly aliasing pointer, which would leave one load in flight
// per lane).
template <int KIND, bool PHASED>
constexpr int kLaneChunks = piece_warp_chunks(KIND, PHASED) / 32;  // chunks per lane

// Source unit of a chunk, per kind: 8 bf16 elements in an aligned 16-byte
// unit, 8 int8 codes in an aligned 8-byte unit, 8 int4 codes in an aligned
// 4-byte unit.  Realignment always moves 8 bf16 values (the copy's units, or
// dequantized ones) by PH elements; the phase is the same for a whole piece,
// hence for a whole warp, so it is compiled per phase: a few funnel shifts
// of fixed words.
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
};

// Exact binary32 value of a code without a conversion instruction: the code
// plus a bias (128 for int8, 8 for int4) is an integer below 2^8; a byte
// permute places byte k of a word of such biased codes in the low mantissa
// bits of 2^23, and subtracting 2^23 + bias is exact.
__device__ __forceinline__ float biased_code_f32(uint32_t byte_word, int k) {
    return __uint_as_float(__byte_perm(byte_word, 0x4B000000u, 0x7650u | static_cast<uint32_t>(k)));
}

// bf16_rne((a - K) * s) and bf16_rne((b - K) * s) as one packed bf16 pair:
// the binary32 subtraction and multiplication, each rounded to nearest even,
// issued as one two-lane instruction each (sub/mul .rn.f32x2).
__device__ __forceinline__ uint32_t dequant_pair(float a, float b, float K, float s) {
    float ya, yb;
    asm("{\n\t.reg .b64 p, k, q;\n\t"
        "mov.b64 p, {%2, %3};\n\tmov.b64 k, {%4, %4};\n\tsub.rn.f32x2 p, p, k;\n\t"
        "mov.b64 q, {%5, %5};\n\tmul.rn.f32x2 p, p, q;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "=f"(ya), "=f"(yb)
        : "f"(a), "f"(b), "f"(K), "f"(s));
    return pack_bf16x2(ya, yb);
}

// The 8 codes of an aligned source unit times their block scale s, as 8
// bf16: y = bf16_rne(f32(code) * s).  Units start at multiples of 8 in the
// shard and blocks at multiples of 256, so one scale serves the whole unit.
template <int KIND>
__device__ __forceinline__ uint4 dequant_unit(const typename Unit<KIND>::T& u, float s) {
    uint32_t w[4];
    if constexpr (KIND == kPieceInt4) {
        // the biased nibbles split once into a word of the even codes (low
        // nibbles) and one of the odd codes (high nibbles), one per byte
        const uint32_t x = u ^ 0x88888888u;
        const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = dequant_pair(biased_code_f32(lo, k), biased_code_f32(hi, k), 8388616.0f, s);  // 2^23 + 8
    } else {
        const uint32_t x0 = u.x ^ 0x80808080u, x1 = u.y ^ 0x80808080u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t x = k < 2 ? x0 : x1;
            w[k] = dequant_pair(biased_code_f32(x, 2 * (k & 1)), biased_code_f32(x, 2 * (k & 1) + 1),
                                8388736.0f, s);  // 2^23 + 128
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
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

// Phase 2 of the copy at source phase PH: take the neighbour's unit by
// shuffle (lane 31 loaded its own), realign and store the vector chunks.
// Every lane of the warp calls this (the shuffles need all of them).
template <int PH>
__device__ __forceinline__ void copy_phase2(uint16_t* dst, int lane, uint4* cur, const uint4* nxt,
                                            const bool* vec) {
    using U = Unit<kPieceBf16>;
#pragma unroll
    for (int j = 0; j < kLaneChunks<kPieceBf16, false>; ++j) {
        uint4 u = cur[j];
        if constexpr (PH != 0) {
            const uint4 n = U::shfl(cur[j]);
            u = U::template realign<PH>(cur[j], lane == 31 ? nxt[j] : n);
        }
        if (!vec[j]) continue;
        *reinterpret_cast<uint4*>(dst + 256 * j) = u;
    }
}

// Phase 2 of a dequantizing piece at source phase PH.  Each lane
// dequantizes its own source units, then the bf16 results are realigned as
// in the copy: a unit never straddles two 256-element scale blocks (a
// realigned chunk can), so every unit takes one scale and no per-element
// select.  A chunk at phase PH needs
// its own unit and the next one: lane l's next unit is lane l + 1's of the
// same step, lane 31's is lane 0's of the next step, and for the last step
// lane 0's extra unit `ext` (the one after the warp's last).  One indexed
// shuffle per word serves both cases: lane 0 offers its next step's value.
template <int KIND, int C, int PH>
__device__ __forceinline__ void dequant_phase2(uint16_t* dst, int lane,
                                               const typename Unit<KIND>::T* cur, const float* sc,
                                               const typename Unit<KIND>::T& ext, float sce,
                                               const bool* vec) {
    if constexpr (PH == 0) {
#pragma unroll
        for (int j = 0; j < C; ++j)
            if (vec[j]) *reinterpret_cast<uint4*>(dst + 256 * j) = dequant_unit<KIND>(cur[j], sc[j]);
    } else {
        // each unit is dequantized just before the chunk that first needs
        // it, so two dequantized units are live at a time
        const int from = (lane + 1) & 31;
        uint4 o = dequant_unit<KIND>(cur[0], sc[0]);
#pragma unroll
        for (int j = 0; j < C; ++j) {
            // lane 0's next unit (the one after the warp's last for j = C-1)
            const uint4 on = j + 1 < C ? dequant_unit<KIND>(cur[j + 1], sc[j + 1])
                                       : dequant_unit<KIND>(ext, sce);
            const uint4 give = lane == 0 ? on : o;
            uint4 n;
            n.x = __shfl_sync(0xffffffffu, give.x, from);
            n.y = __shfl_sync(0xffffffffu, give.y, from);
            n.z = __shfl_sync(0xffffffffu, give.z, from);
            n.w = __shfl_sync(0xffffffffu, give.w, from);
            const uint4 x = Unit<kPieceBf16>::template realign<PH>(o, n);
            if (vec[j]) *reinterpret_cast<uint4*>(dst + 256 * j) = x;
            o = on;
        }
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
    constexpr int C = kLaneChunks<KIND, PHASED>;
    constexpr int kWarpElems = 32 * C * 8;
    const int64_t wbase = static_cast<int64_t>(w - a.warp0[lo]) * kWarpElems;
    const int64_t d00 = wbase + 8 * lane;
    const int64_t x0 = P.s0 + d00;  // its source index
    const char* src = U::at(P.src, x0 - ph);  // the aligned source unit under it
    constexpr int kStep = 32 * U::kUnitBytes;
    bool vec[C];
    uint16_t* dst = P.dst + d00;
    // Phase 1: every load of the vector chunks (source units, block scales).
    // A warp whose chunks and the units around them lie inside the piece
    // (nearly all warps) needs no per-chunk bounds.
    const bool interior = wbase >= P.lo + 8 && wbase + kWarpElems + 8 <= P.hi;
    if constexpr (KIND == kPieceBf16) {
        uint4 cur[C], nxt[C];
        if (interior) {
#pragma unroll
            for (int j = 0; j < C; ++j) {
                vec[j] = true;
                cur[j] = U::load(src + j * kStep);
                if (PHASED && ph && lane == 31) nxt[j] = U::load(src + j * kStep + U::kUnitBytes);
            }
        } else {
#pragma unroll
            for (int j = 0; j < C; ++j) {
                // the source unit under the chunk starts at destination index b
                const int64_t b = d00 + 256 * j - ph;
                vec[j] = b >= P.lo && b + (ph ? 16 : 8) <= P.hi;
                if (b >= P.lo && b + 8 <= P.hi) cur[j] = U::load(src + j * kStep);
                if (PHASED && ph && lane == 31 && vec[j])
                    nxt[j] = U::load(src + j * kStep + U::kUnitBytes);
            }
        }
        // Phase 2: realign (per phase, warp-uniform) and store.
        if constexpr (!PHASED) {
            copy_phase2<0>(dst, lane, cur, nxt, vec);
        } else {
            switch (ph) {
                case 0: copy_phase2<0>(dst, lane, cur, nxt, vec); break;
                case 1: copy_phase2<1>(dst, lane, cur, nxt, vec); break;
                case 2: copy_phase2<2>(dst, lane, cur, nxt, vec); break;
                case 3: copy_phase2<3>(dst, lane, cur, nxt, vec); break;
                case 4: copy_phase2<4>(dst, lane, cur, nxt, vec); break;
                case 5: copy_phase2<5>(dst, lane, cur, nxt, vec); break;
                case 6: copy_phase2<6>(dst, lane, cur, nxt, vec); break;
                default: copy_phase2<7>(dst, lane, cur, nxt, vec); break;
            }
        }
    } else {
        // The lane's units at steps 0..3 start at source index xu + 256 j
        // (xu is negative on some edge lanes, never where a unit is read);
        // lane 0 also reads the unit after the warp's last when phased.
        typename U::T cur[C], ext = {};
        float sc[C], sce = 0.0f;
        const int64_t xu = x0 - ph;
        const bool want_ext = PHASED && ph != 0 && lane == 0;
        if (interior) {
            const float* sp = P.scales + static_cast<uint64_t>(xu) / kQwzBlock;  // xu > 0 here
#pragma unroll
            for (int j = 0; j < C; ++j) {
                vec[j] = true;
                cur[j] = U::load(src + j * kStep);
                sc[j] = sp[j];
            }
            if (want_ext) {
                ext = U::load(src + C * kStep);
                sce = sp[C];
            }
        } else {
#pragma unroll
            for (int j = 0; j < C; ++j) {
                const int64_t b = d00 + 256 * j - ph;  // destination index of the unit's start
                vec[j] = b >= P.lo && b + (ph ? 16 : 8) <= P.hi;
                cur[j] = typename U::T{};
                sc[j] = 0.0f;
                if (b >= P.lo && b + 8 <= P.hi) {
                    cur[j] = U::load(src + j * kStep);
                    sc[j] = P.scales[static_cast<uint64_t>(xu + 256 * j) / kQwzBlock];
                }
            }
            if (want_ext) {
                const int64_t b = d00 + 256 * C - ph;
                if (b >= P.lo && b + 8 <= P.hi) {
                    ext = U::load(src + C * kStep);
                    sce = P.scales[static_cast<uint64_t>(xu + 256 * C) / kQwzBlock];
                }
            }
        }
        if constexpr (!PHASED) {
            dequant_phase2<KIND, C, 0>(dst, lane, cur, sc, ext, sce, vec);
        } else {
            switch (ph) {
                case 0: dequant_phase2<KIND, C, 0>(dst, lane, cur, sc, ext, sce, vec); break;
                case 1: dequant_phase2<KIND, C, 1>(dst, lane, cur, sc, ext, sce, vec); break;
                case 2: dequant_phase2<KIND, C, 2>(dst, lane, cur, sc, ext, sce, vec); break;
                case 3: dequant_phase2<KIND, C, 3>(dst, lane, cur, sc, ext, sce, vec); break;
                case 4: dequant_phase2<KIND, C, 4>(dst, lane, cur, sc, ext, sce, vec); break;
                case 5: dequant_phase2<KIND, C, 5>(dst, lane, cur, sc, ext, sce, vec); break;
                case 6: dequant_phase2<KIND, C, 6>(dst, lane, cur, sc, ext, sce, vec); break;
                default: dequant_phase2<KIND, C, 7>(dst, lane, cur, sc, ext, sce, vec); break;
            }
        }
    }
    // Phase 3: the chunks at the piece's edges, element by element.  Kept out
    // of the load phase: with its stores between the loads, the loads of the
    // later chunks were no longer all in flight together (measured: the int8
    // dequantizing all-gather at 1.3B took 0.84 ms instead of 0.66 ms).
    // A rolled loop over a mask of the lane's remaining chunks: unrolled, it
    // kept phase 2's values alive across it and spilled.
    if (!interior) {
        uint32_t todo = 0;
#pragma unroll
        for (int j = 0; j < C; ++j) todo |= vec[j] ? 0u : 1u << j;
        while (todo) {
            const int j = __ffs(todo) - 1;
            todo &= todo - 1;
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
