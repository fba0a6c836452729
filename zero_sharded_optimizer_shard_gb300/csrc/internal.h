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
    kGather = 3,   // sparam -> full
    kCast = 4,     // master -> sparam (+ full)
    kFusedRep = 5, // grads -> reduce -> AdamW -> every rank's full copy (ZeRO-1/2)
    kFusedQ = 6,   // grads -> reduce -> AdamW -> sparam + int8 codes/scales (qwZ)
    kQuant = 7,    // sparam -> int8 codes/scales (qwZ)
    kDequant = 8,  // int8 codes/scales -> full (qwZ all-gather)
};

// qwZ block: one warp's 32 chunks of 8 elements.
constexpr int kQwzBlock = 256;

constexpr int kMaxSpans = ZERO3_MAX_RANKS;

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
    const void* in;      // shard grad (kAdam) or sparam (kGather, kQuant) or master (kCast)
    int8_t* codes;       // qwZ codes of the shard (kFusedQ, kQuant out; kDequant in)
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

// Gather of submodule segments into a contiguous output.
constexpr int kMaxGatherSegs = 64;
struct GatherSeg {
    const uint16_t* src;   // element 0 of the piece
    int64_t dst_off;       // offset of the piece in out
    int64_t len;
    int64_t chunk0;
    int32_t sphase;        // element phase of the source at an aligned chunk of out
    int32_t pad_;
};
struct GatherArgs {
    uint16_t* out;
    GatherSeg seg[kMaxGatherSegs];
    int64_t total_chunks;
    int32_t n_segs;
    int32_t pad_;
};

cudaError_t launch_stream(int mode, const StreamArgs& a, cudaStream_t stream);

// Submodule gather shared by zero3_fetch_submodule and the prefetch
// coordinator: validation of the sources, and the launches (one per 64
// pieces) writing submodule k's tensors contiguously into out.
zero3_status check_gather_sources(const zero3_plan* p, int32_t k, const uint16_t* const* sparam,
                                  const uint16_t* persist_param, const uint16_t* out);
zero3_status gather_submodule(const zero3_plan* p, int32_t k, const uint16_t* const* sparam,
                              const uint16_t* persist_param, uint16_t* out, cudaStream_t stream);
cudaError_t launch_gather(const GatherArgs& a, cudaStream_t stream);

}  // namespace z3
