// Internal declarations shared by the planner, the C ABI and the kernels.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/zero3.h"

struct zero3_plan {
    int32_t n_ranks = 1;
    int64_t threshold = 0;
    int64_t bucket = 1;
    std::vector<int64_t> numel;
    std::vector<int32_t> submodule;
    std::vector<uint8_t> persistent;
    std::vector<int64_t> offset;
    int64_t n_partitioned = 0;
    int64_t psi_p = 0, psi_pad = 0, S = 0, psi_s = 0;
    // segments of every tensor, concatenated; seg_begin[t]..seg_begin[t+1]
    std::vector<zero3_segment> segs;
    std::vector<int64_t> seg_begin;
    // submodules: member tensors in list order
    std::vector<std::vector<int64_t>> sub_tensors;
    std::vector<int64_t> sub_numel;
    // parameter state machine per submodule
    std::vector<int32_t> status;
    std::vector<int32_t> refs;
    std::vector<uint16_t*> fetched_out;
    std::vector<cudaEvent_t> events;
};

namespace z3 {

// binary32 scalars of one AdamW step
struct Scalars {
    float decay, b1, omb1, b2, omb2, inv_sqrt_bc2, eps, step_size, inv_nd;
};

Scalars make_scalars(const zero3_adamw_hparams& hp, int64_t t, int32_t n_ranks);

// Kernel modes of the streaming kernel.
enum Mode : int {
    kFused = 0,    // grads -> reduce -> AdamW -> sparam (+ full)
    kReduce = 1,   // grads -> reduce -> shard grad (bf16 or f32)
    kAdam = 2,     // shard grad -> AdamW -> sparam
    kCast = 4,     // master -> sparam (+ full)
    kFusedRep = 5, // grads -> reduce -> AdamW -> every rank's full copy (ZeRO-1/2)
    kFusedQ = 6,   // grads -> reduce -> AdamW -> sparam + int8 codes/scales (qwZ)
    kQuant = 7,    // sparam -> int8 codes/scales (qwZ)
};

// qwZ block: one warp's 32 chunks of 8 elements.
constexpr int kQwzBlock = 256;

// one span per owning rank, plus the persistent group in the fused step
constexpr int kMaxSpans = ZERO3_MAX_RANKS + 1;

// One owner's slice of the requested range: local indices [lo, hi).
struct Span {
    int64_t lo, hi;
    int64_t gofs;        // grads element offset of local index 0 (grads[q] + gofs + i)
    int64_t fofs;        // full element offset of local index 0, or -1 (no full write)
    int64_t chunk0;      // first 8-element chunk of this span in the launch's chunk space
    float* master;
    float* m;
    float* v;
    void* out;           // sparam (bf16) or shard grad (kReduce)
    const void* in;      // shard grad (kAdam) or sparam (kQuant) or master (kCast)
    int8_t* codes;       // qwZ codes of the shard (kFusedQ, kQuant out)
    float* scales;       // qwZ block scales of the shard
    // Element phase (address / 2 mod 8) of the gradient and all-gather
    // streams at local index 0; states and shards are always 16-byte aligned
    // at multiples of 8.  Interior chunks load/store the phased streams at
    // the widest aligned width (16, 8, 4 or 2 bytes).
    int32_t gphase;
    int32_t fphase;
};

struct StreamArgs {
    const uint16_t* grads[ZERO3_MAX_RANKS];
    uint16_t* reps[ZERO3_MAX_RANKS];   // kFusedRep: every rank's full parameter copy
    uint16_t* full;
    Span span[kMaxSpans];
    int64_t total_chunks;
    int32_t n_spans;
    int32_t nd;
    int32_t dtype;       // zero3_dtype of the shard grad (kReduce out / kAdam in); qwZ bits
    int32_t pad_;
    Scalars sc;
};

// Copy-like launches (submodule gathers, the all-gather copy, the
// dequantizing all-gather) are lists of pieces.  A piece writes destination
// elements [lo, hi) of `dst`, which is 16-byte aligned (lo < 8), and element
// d comes from source index s0 + d: a bf16 value of `src`, or a qwZ code of
// the shard `src` with its block scale scales[(s0 + d) / 256].  The
// destination is cut into 8-element chunks aligned to `dst`, and the source
// of a chunk starts at phase `ph`: in elements (bf16), bytes (int8 codes) or
// nibbles (int4 codes) past an aligned unit.
enum PieceKind : int { kPieceBf16 = 16, kPieceInt8 = 8, kPieceInt4 = 4 };

struct Piece {
    const void* src;
    const float* scales;
    uint16_t* dst;
    int64_t s0;
    int64_t lo, hi;
    int32_t ph;
    int32_t pad_;
};

// A warp takes consecutive chunks of one piece: 128 (1024 elements), or 192
// in a dequantizing launch where some source is phased (such a warp's
// per-warp set-up and its one extra source unit then weigh less per chunk;
// its units are 8 or 4 bytes, so six per lane fit the registers).  The
// launch's warps are numbered piece after piece.  warp0[i] is the first warp
// of piece i and warp0[n] the launch's warp count, so the piece of a warp is
// found by a binary search that every lane of the warp takes alike.
constexpr int piece_warp_chunks(int kind, bool phased) {
    return kind != kPieceBf16 && phased ? 192 : 128;
}
constexpr int kSmallPieces = 64;    // one submodule, the all-gathers
constexpr int kLargePieces = 512;   // several submodules in one launch
template <int MAXP>
struct PieceArgs {
    uint32_t warp0[MAXP + 1];
    int32_t n;
    int32_t pad_;
    Piece piece[MAXP];
};

// Builds piece launches and issues one whenever the description is full
// (or the warp count would overflow its 32-bit numbering).
class PieceLauncher {
  public:
    PieceLauncher(int kind, cudaStream_t stream, bool large);
    ~PieceLauncher();
    PieceLauncher(const PieceLauncher&) = delete;
    PieceLauncher& operator=(const PieceLauncher&) = delete;
    // Appends the piece writing dst[i] for i in [0, len) from source index
    // src_index + i; `dst` need not be aligned (the piece starts at its
    // phase).  `src` is the source buffer (bf16 elements or codes of a shard,
    // 16-byte aligned).  ZERO3_ENOMEM if the description could not be
    // allocated, ZERO3_ECUDA if a launch failed.
    zero3_status add(const void* src, const float* scales, int64_t src_index, uint16_t* dst,
                     int64_t len);
    // Launches what has been added so far.
    zero3_status flush();
    int64_t launches() const { return launches_; }

  private:
    int kind_;
    cudaStream_t stream_;
    bool large_;
    void* args_;   // PieceArgs<kSmallPieces> or PieceArgs<kLargePieces>
    int64_t launches_ = 0;
};

cudaError_t launch_stream(int mode, const StreamArgs& a, cudaStream_t stream);
cudaError_t launch_pieces_small(int kind, const PieceArgs<kSmallPieces>& a, cudaStream_t stream);
cudaError_t launch_pieces_large(int kind, const PieceArgs<kLargePieces>& a, cudaStream_t stream);

// Submodule gathers shared by zero3_fetch_submodule(s) and the prefetch
// coordinator: validation of the sources, and the launches writing each
// submodule's tensors contiguously into its output.
zero3_status check_gather_sources(const zero3_plan* p, int32_t k, const uint16_t* const* sparam,
                                  const uint16_t* persist_param, const uint16_t* out);
// Gathers submodules ks[0..n) into outs[0..n) with as few launches as the
// piece limit allows.  Sources and outputs must have been checked.
zero3_status gather_submodules(const zero3_plan* p, const int32_t* ks, int64_t n,
                               const uint16_t* const* sparam, const uint16_t* persist_param,
                               uint16_t* const* outs, cudaStream_t stream,
                               int64_t* n_launches = nullptr);

}  // namespace z3
