// C ABI of the compute calls: argument checks, the per-rank spans of a flat
// range, the submodule state machine, and the launches.
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "internal.h"

namespace {

using z3::Span;
using z3::StreamArgs;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool range_ok(const zero3_plan* p, int64_t lo, int64_t hi) {
    return 0 <= lo && lo <= hi && hi <= p->psi_pad;
}

bool hparams_ok(const zero3_adamw_hparams* hp, int64_t t) {
    if (!hp || t < 1) return false;
    const double v[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (double x : v)
        if (!std::isfinite(x)) return false;
    return hp->beta1 >= 0.0 && hp->beta1 < 1.0 && hp->beta2 >= 0.0 && hp->beta2 < 1.0 &&
           hp->lr >= 0.0 && hp->eps >= 0.0;
}

zero3_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ZERO3_OK : ZERO3_ECUDA; }

// Checks the N_d gradient pointers: present and 16-byte aligned.
bool grads_ok(const zero3_plan* p, const uint16_t* const* grads) {
    if (!grads) return false;
    for (int q = 0; q < p->n_ranks; ++q)
        if (!grads[q] || !aligned16(grads[q])) return false;
    return true;
}

// Local range of rank r inside flat [lo, hi); empty when b <= a.
void rank_range(const zero3_plan* p, int r, int64_t lo, int64_t hi, int64_t* a, int64_t* b) {
    const int64_t s0 = static_cast<int64_t>(r) * p->S, s1 = s0 + p->S;
    *a = (lo > s0 ? lo : s0) - s0;
    *b = (hi < s1 ? hi : s1) - s0;
}

// Appends a span and advances the chunk counter.  With warp_blocks, the
// span's chunks start on a multiple of 32 so that each warp covers exactly
// one 256-element qwZ block (the span then starts on a block boundary).
void add_span(StreamArgs& a, Span s, bool warp_blocks = false) {
    const int64_t first = s.lo & ~static_cast<int64_t>(7);
    if (warp_blocks) a.total_chunks = (a.total_chunks + 31) / 32 * 32;
    s.chunk0 = a.total_chunks;
    a.span[a.n_spans++] = s;
    a.total_chunks += (s.hi - first + 7) / 8;
    if (warp_blocks) a.total_chunks = (a.total_chunks + 31) / 32 * 32;
}

struct RankPtrs {
    const uint16_t* const* grads = nullptr;
    int64_t grads_origin = 0;
    float* const* master = nullptr;
    float* const* m = nullptr;
    float* const* v = nullptr;
    void* const* out = nullptr;        // sparam or shard grad
    const void* const* in = nullptr;   // shard grad, sparam or master
    uint16_t* full = nullptr;
    int8_t* const* codes = nullptr;    // qwZ codes per rank
    float* const* scales = nullptr;    // qwZ scales per rank
    bool need_state = false;
    bool warp_blocks = false;          // quantizing launch: one warp per 256-element block
};

// Builds the launch description of one mode over flat [lo, hi).  Validates
// the pointers of every rank that owns part of the range.
zero3_status build_args(const zero3_plan* p, int mode, const RankPtrs& rp, int64_t lo, int64_t hi,
                        const z3::Scalars* sc, int dtype, StreamArgs& a) {
    std::memset(&a, 0, sizeof(a));
    a.nd = p->n_ranks;
    a.dtype = dtype;
    a.full = rp.full;
    if (sc) a.sc = *sc;
    if (rp.grads)
        for (int q = 0; q < p->n_ranks; ++q) a.grads[q] = rp.grads[q];
    for (int r = 0; r < p->n_ranks; ++r) {
        int64_t la, lb;
        rank_range(p, r, lo, hi, &la, &lb);
        if (lb <= la) continue;
        Span s;
        std::memset(&s, 0, sizeof(s));
        s.lo = la;
        s.hi = lb;
        if (rp.grads) {
            s.gofs = static_cast<int64_t>(r) * p->S - rp.grads_origin;
            s.gphase = static_cast<int32_t>(s.gofs & 7);  // two's complement: also for gofs < 0
        }
        if (rp.full) {
            s.fofs = static_cast<int64_t>(r) * p->S;
            s.fphase = static_cast<int32_t>(s.fofs & 7);
        } else {
            s.fofs = -1;
        }
        if (rp.need_state) {
            if (!rp.master || !rp.m || !rp.v) return ZERO3_EINVAL;
            s.master = rp.master[r];
            s.m = rp.m[r];
            s.v = rp.v[r];
            if (!s.master || !s.m || !s.v) return ZERO3_EINVAL;
            if (!aligned16(s.master) || !aligned16(s.m) || !aligned16(s.v)) return ZERO3_EINVAL;
        }
        if (rp.out) {
            s.out = rp.out[r];
            if (!s.out || !aligned16(s.out)) return ZERO3_EINVAL;
        }
        if (rp.in) {
            s.in = rp.in[r];
            if (!s.in || !aligned16(s.in)) return ZERO3_EINVAL;
        }
        if (rp.codes) {
            s.codes = rp.codes[r];
            s.scales = rp.scales ? rp.scales[r] : nullptr;
            if (!s.codes || !aligned16(s.codes) || !s.scales || !aligned16(s.scales))
                return ZERO3_EINVAL;
        }
        if (rp.warp_blocks) {
            // a quantizing launch covers whole blocks of each shard
            if (la % z3::kQwzBlock != 0 || (lb % z3::kQwzBlock != 0 && lb != p->S))
                return ZERO3_EINVAL;
        }
        add_span(a, s, rp.warp_blocks);
    }
    return ZERO3_OK;
}

z3::Scalars step_scalars(const zero3_plan* p, const zero3_adamw_hparams* hp, int64_t t) {
    return z3::make_scalars(*hp, t, p->n_ranks);
}

bool persist_ok(const zero3_plan* p, const zero3_persist_state* ps) {
    if (p->psi_s == 0) return true;
    return ps && grads_ok(p, ps->grads) && ps->master && ps->m && ps->v && ps->param &&
           aligned16(ps->master) && aligned16(ps->m) && aligned16(ps->v) && aligned16(ps->param);
}

// The persistent group as one span of a fused launch: local indices
// [0, psi_s) of its resident copy, no write to `full`, gradients at element
// offset gofs from the launch's gradient pointers (the arithmetic per element
// is the flat spans').
void add_persistent_span(const zero3_plan* p, const zero3_persist_state* ps, int64_t gofs,
                         StreamArgs& a) {
    Span s;
    std::memset(&s, 0, sizeof(s));
    s.lo = 0;
    s.hi = p->psi_s;
    s.gofs = gofs;
    s.gphase = static_cast<int32_t>(gofs & 7);  // two's complement: also for gofs < 0
    s.fofs = -1;
    s.master = ps->master;
    s.m = ps->m;
    s.v = ps->v;
    s.out = ps->param;
    add_span(a, s);
}

// When every rank's persistent-group gradient sits at the same element
// offset from that rank's flat gradient pointer (for instance right after the
// flat gradients in one buffer per rank), returns true and the offset: the
// group can then ride in the flat launch as one more span.
bool common_persist_offset(const zero3_plan* p, const uint16_t* const* grads,
                           const zero3_persist_state* ps, int64_t* gofs) {
    if (!grads || !ps || !ps->grads) return false;
    int64_t d0 = 0;
    for (int q = 0; q < p->n_ranks; ++q) {
        if (!grads[q] || !ps->grads[q]) return false;
        const int64_t d = static_cast<int64_t>(reinterpret_cast<uintptr_t>(ps->grads[q]) -
                                               reinterpret_cast<uintptr_t>(grads[q]));
        if (d % 2 != 0 || (q > 0 && d != d0)) return false;
        d0 = d;
    }
    *gofs = d0 / 2;
    return true;
}

zero3_status persistent_launch(const zero3_plan* p, const z3::Scalars& sc,
                               const zero3_persist_state* ps, cudaStream_t stream) {
    if (p->psi_s == 0) return ZERO3_OK;
    if (!persist_ok(p, ps)) return ZERO3_EINVAL;
    StreamArgs a;
    std::memset(&a, 0, sizeof(a));
    a.nd = p->n_ranks;
    a.sc = sc;
    for (int q = 0; q < p->n_ranks; ++q) a.grads[q] = ps->grads[q];
    add_persistent_span(p, ps, 0, a);
    return cuda_status(z3::launch_stream(z3::kFused, a, stream));
}

}  // namespace

namespace z3 {

zero3_status check_gather_sources(const zero3_plan* p, int32_t k, const uint16_t* const* sparam,
                                  const uint16_t* persist_param, const uint16_t* out) {
    if (p->sub_numel[k] > 0 && (!out || !aligned16(out))) return ZERO3_EINVAL;
    for (int64_t t : p->sub_tensors[k]) {
        if (p->numel[t] == 0) continue;
        if (p->persistent[t]) {
            if (!persist_param || !aligned16(persist_param)) return ZERO3_EINVAL;
        } else {
            if (!sparam) return ZERO3_EINVAL;
            for (int64_t s = p->seg_begin[t]; s < p->seg_begin[t + 1]; ++s) {
                const uint16_t* src = sparam[p->segs[s].rank];
                if (!src || !aligned16(src)) return ZERO3_EINVAL;
            }
        }
    }
    return ZERO3_OK;
}

PieceLauncher::PieceLauncher(int kind, cudaStream_t stream, bool large)
    : kind_(kind), stream_(stream), large_(large) {
    if (large) {
        auto* a = new (std::nothrow) PieceArgs<kLargePieces>;
        if (a) a->n = 0;
        args_ = a;
    } else {
        auto* a = new (std::nothrow) PieceArgs<kSmallPieces>;
        if (a) a->n = 0;
        args_ = a;
    }
}

PieceLauncher::~PieceLauncher() {
    if (large_)
        delete static_cast<PieceArgs<kLargePieces>*>(args_);
    else
        delete static_cast<PieceArgs<kSmallPieces>*>(args_);
}

namespace {

template <int MAXP>
zero3_status piece_flush(PieceArgs<MAXP>& a, int kind, cudaStream_t stream, int64_t* launches,
                         cudaError_t (*launch)(int, const PieceArgs<MAXP>&, cudaStream_t)) {
    if (a.n == 0) return ZERO3_OK;
    // pieces were numbered at 128 chunks per warp; a phased dequantizing
    // launch takes more per warp (fewer warps, so the 32-bit bound holds)
    bool phased = false;
    for (int i = 0; i < a.n; ++i) phased = phased || a.piece[i].ph != 0;
    const uint64_t wc = static_cast<uint64_t>(piece_warp_chunks(kind, phased));
    if (wc != 128) {
        for (int i = 0; i < a.n; ++i) {
            const uint64_t chunks = static_cast<uint64_t>((a.piece[i].hi + 7) / 8);
            a.warp0[i + 1] = a.warp0[i] + static_cast<uint32_t>((chunks + wc - 1) / wc);
        }
    }
    const cudaError_t e = launch(kind, a, stream);
    a.n = 0;
    if (e != cudaSuccess) return ZERO3_ECUDA;
    *launches += 1;
    return ZERO3_OK;
}

// Appends one piece; flushes first when the description is full or the
// launch's warp count would not fit its 32-bit numbering.
template <int MAXP>
zero3_status piece_add(PieceArgs<MAXP>& a, int kind, cudaStream_t stream, int64_t* launches,
                       cudaError_t (*launch)(int, const PieceArgs<MAXP>&, cudaStream_t),
                       const Piece& pc) {
    const uint64_t chunks = static_cast<uint64_t>((pc.hi + 7) / 8);
    const uint64_t wc = static_cast<uint64_t>(piece_warp_chunks(kind, false));
    const uint64_t warps = (chunks + wc - 1) / wc;
    const uint64_t cap = 0xffffffffull - 256;  // room for the grid rounding
    if (warps > cap) return ZERO3_EINVAL;  // a single piece beyond 2^41 elements
    if (a.n == MAXP || (a.n > 0 && a.warp0[a.n] + warps > cap)) {
        zero3_status st = piece_flush(a, kind, stream, launches, launch);
        if (st != ZERO3_OK) return st;
    }
    if (a.n == 0) a.warp0[0] = 0;
    a.piece[a.n] = pc;
    a.warp0[a.n + 1] = a.warp0[a.n] + static_cast<uint32_t>(warps);
    a.n += 1;
    return ZERO3_OK;
}

}  // namespace

zero3_status PieceLauncher::add(const void* src, const float* scales, int64_t src_index,
                                uint16_t* dst, int64_t len) {
    if (!args_) return ZERO3_ENOMEM;
    if (len <= 0) return ZERO3_OK;
    // destination base rounded down to 16 bytes; the piece starts at lo
    const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
    const int64_t lo = static_cast<int64_t>((da >> 1) & 7u);
    Piece pc;
    std::memset(&pc, 0, sizeof(pc));
    pc.src = src;
    pc.scales = scales;
    pc.dst = dst - lo;
    pc.lo = lo;
    pc.hi = lo + len;
    pc.s0 = src_index - lo;
    if (kind_ == kPieceBf16)  // element phase of the source at aligned destination chunks
        pc.ph = static_cast<int32_t>(
            (static_cast<int64_t>(reinterpret_cast<uintptr_t>(src) >> 1) + pc.s0) & 7);
    else  // code buffers are 16-byte aligned: the phase is the source index's
        pc.ph = static_cast<int32_t>(pc.s0 & 7);
    if (large_)
        return piece_add(*static_cast<PieceArgs<kLargePieces>*>(args_), kind_, stream_,
                         &launches_, launch_pieces_large, pc);
    return piece_add(*static_cast<PieceArgs<kSmallPieces>*>(args_), kind_, stream_, &launches_,
                     launch_pieces_small, pc);
}

zero3_status PieceLauncher::flush() {
    if (!args_) return ZERO3_ENOMEM;
    if (large_)
        return piece_flush(*static_cast<PieceArgs<kLargePieces>*>(args_), kind_, stream_,
                           &launches_, launch_pieces_large);
    return piece_flush(*static_cast<PieceArgs<kSmallPieces>*>(args_), kind_, stream_, &launches_,
                       launch_pieces_small);
}

// Pieces of submodule k: each member tensor in list order, a persistent one
// from its resident copy, a partitioned one segment by segment from the
// owning shards.
int64_t submodule_pieces(const zero3_plan* p, int32_t k) {
    int64_t n = 0;
    for (int64_t t : p->sub_tensors[k]) {
        if (p->numel[t] == 0) continue;
        n += p->persistent[t] ? 1 : p->seg_begin[t + 1] - p->seg_begin[t];
    }
    return n;
}

zero3_status gather_submodules(const zero3_plan* p, const int32_t* ks, int64_t n,
                               const uint16_t* const* sparam, const uint16_t* persist_param,
                               uint16_t* const* outs, cudaStream_t stream, int64_t* n_launches) {
    int64_t pieces = 0;
    for (int64_t i = 0; i < n; ++i) pieces += submodule_pieces(p, ks[i]);
    PieceLauncher L(kPieceBf16, stream, pieces > kSmallPieces);
    for (int64_t i = 0; i < n; ++i) {
        const int32_t k = ks[i];
        uint16_t* out = outs[i];
        int64_t running = 0;
        for (int64_t t : p->sub_tensors[k]) {
            zero3_status st = ZERO3_OK;
            if (p->persistent[t]) {
                st = L.add(persist_param, nullptr, p->offset[t], out + running, p->numel[t]);
            } else {
                for (int64_t s = p->seg_begin[t]; s < p->seg_begin[t + 1] && st == ZERO3_OK; ++s) {
                    const zero3_segment& sg = p->segs[s];
                    st = L.add(sparam[sg.rank], nullptr, sg.shard_off, out + running + sg.tensor_off,
                               sg.len);
                }
            }
            if (st != ZERO3_OK) return st;
            running += p->numel[t];
        }
    }
    zero3_status st = L.flush();
    if (n_launches) *n_launches = L.launches();
    return st;
}

}  // namespace z3

extern "C" {

zero3_status zero3_reduce_scatter(const zero3_plan* p, const uint16_t* const* grads,
                                  int64_t grads_origin, int64_t lo, int64_t hi,
                                  void* const* shard_grad, zero3_dtype out_dtype,
                                  zero3_stream stream) {
    if (!p || !range_ok(p, lo, hi) || grads_origin > lo) return ZERO3_EINVAL;
    if (out_dtype != ZERO3_BF16 && out_dtype != ZERO3_F32) return ZERO3_EINVAL;
    if (lo == hi) return ZERO3_OK;
    if (!grads_ok(p, grads) || !shard_grad) return ZERO3_EINVAL;
    RankPtrs rp;
    rp.grads = grads;
    rp.grads_origin = grads_origin;
    rp.out = shard_grad;
    z3::Scalars sc;
    std::memset(&sc, 0, sizeof(sc));
    sc.inv_nd = static_cast<float>(1.0 / static_cast<double>(p->n_ranks));
    StreamArgs a;
    zero3_status st = build_args(p, z3::kReduce, rp, lo, hi, &sc, out_dtype, a);
    if (st != ZERO3_OK) return st;
    return cuda_status(z3::launch_stream(z3::kReduce, a, stream));
}

zero3_status zero3_adamw_step(const zero3_plan* p, const zero3_adamw_hparams* hp, int64_t t,
                              const void* const* shard_grad, zero3_dtype grad_dtype,
                              float* const* master, float* const* m, float* const* v,
                              uint16_t* const* sparam, int64_t lo, int64_t hi,
                              zero3_stream stream) {
    if (!p || !range_ok(p, lo, hi) || !hparams_ok(hp, t)) return ZERO3_EINVAL;
    if (grad_dtype != ZERO3_BF16 && grad_dtype != ZERO3_F32) return ZERO3_EINVAL;
    if (lo == hi) return ZERO3_OK;
    if (!shard_grad || !sparam) return ZERO3_EINVAL;
    RankPtrs rp;
    rp.master = master;
    rp.m = m;
    rp.v = v;
    rp.need_state = true;
    rp.out = reinterpret_cast<void* const*>(sparam);
    rp.in = shard_grad;
    const z3::Scalars sc = step_scalars(p, hp, t);
    StreamArgs a;
    zero3_status st = build_args(p, z3::kAdam, rp, lo, hi, &sc, grad_dtype, a);
    if (st != ZERO3_OK) return st;
    return cuda_status(z3::launch_stream(z3::kAdam, a, stream));
}

zero3_status zero3_allgather(const zero3_plan* p, const uint16_t* const* sparam, uint16_t* full,
                             int64_t lo, int64_t hi, zero3_stream stream) {
    if (!p || !range_ok(p, lo, hi)) return ZERO3_EINVAL;
    if (lo == hi) return ZERO3_OK;
    if (!sparam || !full || !aligned16(full)) return ZERO3_EINVAL;
    for (int r = 0; r < p->n_ranks; ++r) {
        int64_t la, lb;
        rank_range(p, r, lo, hi, &la, &lb);
        if (lb > la && (!sparam[r] || !aligned16(sparam[r]))) return ZERO3_EINVAL;
    }
    // one piece per owning rank: full[r*S + i] = sparam[r][i]
    z3::PieceLauncher L(z3::kPieceBf16, stream, false);
    for (int r = 0; r < p->n_ranks; ++r) {
        int64_t la, lb;
        rank_range(p, r, lo, hi, &la, &lb);
        if (lb <= la) continue;
        zero3_status st = L.add(sparam[r], nullptr, la, full + static_cast<int64_t>(r) * p->S + la,
                                lb - la);
        if (st != ZERO3_OK) return st;
    }
    return L.flush();
}

zero3_status zero3_step(const zero3_plan* p, const zero3_adamw_hparams* hp, int64_t t,
                        const uint16_t* const* grads, int64_t grads_origin, float* const* master,
                        float* const* m, float* const* v, uint16_t* const* sparam,
                        uint16_t* full, const zero3_persist_state* persist, int64_t lo,
                        int64_t hi, zero3_stream stream) {
    if (!p || !range_ok(p, lo, hi) || !hparams_ok(hp, t) || grads_origin > lo)
        return ZERO3_EINVAL;
    const z3::Scalars sc = step_scalars(p, hp, t);
    const bool with_persist = persist && p->psi_s > 0;
    int64_t pofs = 0;
    const bool fold = with_persist && lo < hi && common_persist_offset(p, grads, persist, &pofs);
    // validate the persistent group before the first launch so that an
    // error launches nothing
    if (with_persist) {
        if (!persist->master || !persist->m || !persist->v || !persist->param ||
            !aligned16(persist->master) || !aligned16(persist->m) || !aligned16(persist->v) ||
            !aligned16(persist->param))
            return ZERO3_EINVAL;
        if (!fold && !persist_ok(p, persist)) return ZERO3_EINVAL;
    }
    if (lo < hi) {
        if (!grads_ok(p, grads) || !sparam || !full || !aligned16(full)) return ZERO3_EINVAL;
        RankPtrs rp;
        rp.grads = grads;
        rp.grads_origin = grads_origin;
        rp.master = master;
        rp.m = m;
        rp.v = v;
        rp.need_state = true;
        rp.out = reinterpret_cast<void* const*>(sparam);
        rp.full = full;
        StreamArgs a;
        zero3_status st = build_args(p, z3::kFused, rp, lo, hi, &sc, 0, a);
        if (st != ZERO3_OK) return st;
        // the persistent group rides in the same launch as one more span
        if (fold) add_persistent_span(p, persist, pofs, a);
        st = cuda_status(z3::launch_stream(z3::kFused, a, stream));
        if (st != ZERO3_OK || fold) return st;
    }
    if (with_persist) return persistent_launch(p, sc, persist, stream);
    return ZERO3_OK;
}

zero3_status zero3_step_stage12(const zero3_plan* p, const zero3_adamw_hparams* hp, int64_t t,
                                const uint16_t* const* grads, int64_t grads_origin,
                                float* const* master, float* const* m, float* const* v,
                                uint16_t* const* params, int64_t lo, int64_t hi,
                                zero3_stream stream) {
    if (!p || !range_ok(p, lo, hi) || !hparams_ok(hp, t) || grads_origin > lo)
        return ZERO3_EINVAL;
    if (lo == hi) return ZERO3_OK;
    if (!grads_ok(p, grads) || !params) return ZERO3_EINVAL;
    for (int q = 0; q < p->n_ranks; ++q)
        if (!params[q] || !aligned16(params[q])) return ZERO3_EINVAL;
    const z3::Scalars sc = step_scalars(p, hp, t);
    RankPtrs rp;
    rp.grads = grads;
    rp.grads_origin = grads_origin;
    rp.master = master;
    rp.m = m;
    rp.v = v;
    rp.need_state = true;
    rp.full = params[0];  // every copy has the same layout: offsets and phase
    StreamArgs a;
    zero3_status st = build_args(p, z3::kFusedRep, rp, lo, hi, &sc, 0, a);
    if (st != ZERO3_OK) return st;
    for (int q = 0; q < p->n_ranks; ++q) a.reps[q] = params[q];
    return cuda_status(z3::launch_stream(z3::kFusedRep, a, stream));
}

zero3_status zero3_step_qwz(const zero3_plan* p, const zero3_adamw_hparams* hp, int64_t t,
                            const uint16_t* const* grads, int64_t grads_origin,
                            float* const* master, float* const* m, float* const* v,
                            uint16_t* const* sparam, int32_t bits, int8_t* const* codes,
                            float* const* scales, const zero3_persist_state* persist,
                            int64_t lo, int64_t hi, zero3_stream stream) {
    if (!p || !range_ok(p, lo, hi) || !hparams_ok(hp, t) || grads_origin > lo)
        return ZERO3_EINVAL;
    if (bits != 8 && bits != 4) return ZERO3_EINVAL;
    const z3::Scalars sc = step_scalars(p, hp, t);
    if (lo < hi) {
        if (!grads_ok(p, grads) || !sparam || !codes || !scales) return ZERO3_EINVAL;
        RankPtrs rp;
        rp.grads = grads;
        rp.grads_origin = grads_origin;
        rp.master = master;
        rp.m = m;
        rp.v = v;
        rp.need_state = true;
        rp.out = reinterpret_cast<void* const*>(sparam);
        rp.codes = codes;
        rp.scales = scales;
        rp.warp_blocks = true;
        StreamArgs a;
        zero3_status st = build_args(p, z3::kFusedQ, rp, lo, hi, &sc, bits, a);
        if (st != ZERO3_OK) return st;
        if (persist && !persist_ok(p, persist)) return ZERO3_EINVAL;
        st = cuda_status(z3::launch_stream(z3::kFusedQ, a, stream));
        if (st != ZERO3_OK) return st;
    }
    if (persist) return persistent_launch(p, sc, persist, stream);
    return ZERO3_OK;
}

zero3_status zero3_quantize_shards(const zero3_plan* p, const uint16_t* const* sparam,
                                   int32_t bits, int8_t* const* codes, float* const* scales,
                                   int64_t lo, int64_t hi, zero3_stream stream) {
    if (!p || !range_ok(p, lo, hi)) return ZERO3_EINVAL;
    if (bits != 8 && bits != 4) return ZERO3_EINVAL;
    if (lo == hi) return ZERO3_OK;
    if (!sparam || !codes || !scales) return ZERO3_EINVAL;
    RankPtrs rp;
    rp.in = reinterpret_cast<const void* const*>(sparam);
    rp.codes = codes;
    rp.scales = scales;
    rp.warp_blocks = true;
    StreamArgs a;
    zero3_status st = build_args(p, z3::kQuant, rp, lo, hi, nullptr, bits, a);
    if (st != ZERO3_OK) return st;
    return cuda_status(z3::launch_stream(z3::kQuant, a, stream));
}

zero3_status zero3_allgather_qwz(const zero3_plan* p, int32_t bits, const int8_t* const* codes,
                                 const float* const* scales, uint16_t* full, int64_t lo,
                                 int64_t hi, zero3_stream stream) {
    if (!p || !range_ok(p, lo, hi)) return ZERO3_EINVAL;
    if (bits != 8 && bits != 4) return ZERO3_EINVAL;
    if (lo == hi) return ZERO3_OK;
    if (!codes || !scales || !full || !aligned16(full)) return ZERO3_EINVAL;
    for (int r = 0; r < p->n_ranks; ++r) {
        int64_t la, lb;
        rank_range(p, r, lo, hi, &la, &lb);
        if (lb <= la) continue;
        if (!codes[r] || !aligned16(codes[r]) || !scales[r] || !aligned16(scales[r]))
            return ZERO3_EINVAL;
    }
    // one piece per owning rank: full[r*S + i] = bf16(code_r(i) * scale_r(i / 256))
    z3::PieceLauncher L(bits == 4 ? z3::kPieceInt4 : z3::kPieceInt8, stream, false);
    for (int r = 0; r < p->n_ranks; ++r) {
        int64_t la, lb;
        rank_range(p, r, lo, hi, &la, &lb);
        if (lb <= la) continue;
        zero3_status st = L.add(codes[r], scales[r], la,
                                full + static_cast<int64_t>(r) * p->S + la, lb - la);
        if (st != ZERO3_OK) return st;
    }
    return L.flush();
}

zero3_status zero3_persistent_step(const zero3_plan* p, const zero3_adamw_hparams* hp, int64_t t,
                                   const zero3_persist_state* persist, zero3_stream stream) {
    if (!p || !hparams_ok(hp, t) || !persist) return ZERO3_EINVAL;
    return persistent_launch(p, step_scalars(p, hp, t), persist, stream);
}

zero3_status zero3_cast_params(const zero3_plan* p, const float* const* master,
                               uint16_t* const* sparam, uint16_t* full,
                               const zero3_persist_state* persist, int64_t lo, int64_t hi,
                               zero3_stream stream) {
    if (!p || !range_ok(p, lo, hi)) return ZERO3_EINVAL;
    if (full && !aligned16(full)) return ZERO3_EINVAL;
    if (lo < hi) {
        if (!master || !sparam) return ZERO3_EINVAL;
        RankPtrs rp;
        rp.full = full;
        rp.out = reinterpret_cast<void* const*>(sparam);
        rp.in = reinterpret_cast<const void* const*>(master);
        StreamArgs a;
        zero3_status st = build_args(p, z3::kCast, rp, lo, hi, nullptr, 0, a);
        if (st != ZERO3_OK) return st;
        st = cuda_status(z3::launch_stream(z3::kCast, a, stream));
        if (st != ZERO3_OK) return st;
    }
    if (persist && p->psi_s > 0) {
        if (!persist->master || !persist->param || !aligned16(persist->master) ||
            !aligned16(persist->param))
            return ZERO3_EINVAL;
        StreamArgs a;
        std::memset(&a, 0, sizeof(a));
        a.nd = p->n_ranks;
        Span s;
        std::memset(&s, 0, sizeof(s));
        s.lo = 0;
        s.hi = p->psi_s;
        s.fofs = -1;
        s.in = persist->master;
        s.out = persist->param;
        add_span(a, s);
        return cuda_status(z3::launch_stream(z3::kCast, a, stream));
    }
    return ZERO3_OK;
}

// ------------------------------------------------------------- submodules

zero3_status zero3_fetch_submodule(zero3_plan* p, int32_t k, const uint16_t* const* sparam,
                                   const uint16_t* persist_param, uint16_t* out,
                                   zero3_stream stream) {
    if (!p || k < 0 || k >= static_cast<int32_t>(p->sub_tensors.size())) return ZERO3_EINVAL;
    if (p->status[k] != ZERO3_NOT_AVAILABLE) {
        if (out != p->fetched_out[k]) return ZERO3_ESTATE;
        p->refs[k] += 1;
        return ZERO3_OK;
    }
    zero3_status st = z3::check_gather_sources(p, k, sparam, persist_param, out);
    if (st != ZERO3_OK) return st;
    if (!p->events[k]) {
        if (cudaEventCreateWithFlags(&p->events[k], cudaEventDisableTiming) != cudaSuccess) {
            p->events[k] = nullptr;
            return ZERO3_ECUDA;
        }
    }
    uint16_t* outs[1] = {out};
    st = z3::gather_submodules(p, &k, 1, sparam, persist_param, outs, stream);
    if (st != ZERO3_OK) return st;
    if (cudaEventRecord(p->events[k], stream) != cudaSuccess) return ZERO3_ECUDA;
    p->status[k] = ZERO3_INFLIGHT;
    p->refs[k] = 1;
    p->fetched_out[k] = out;
    return ZERO3_OK;
}

zero3_status zero3_fetch_submodules(zero3_plan* p, const int32_t* ks, int32_t n,
                                    const uint16_t* const* sparam, const uint16_t* persist_param,
                                    uint16_t* const* outs, zero3_stream stream) {
    if (!p || n < 0 || (n > 0 && (!ks || !outs))) return ZERO3_EINVAL;
    const int32_t n_sub = static_cast<int32_t>(p->sub_tensors.size());
    for (int32_t i = 0; i < n; ++i)
        if (ks[i] < 0 || ks[i] >= n_sub) return ZERO3_EINVAL;
    // Walk the list as n single fetches would, on the side: which
    // submodules this call gathers, and the output each one is bound to.
    std::vector<int32_t> gather;
    std::vector<uint16_t*> gather_out;
    std::vector<uint8_t> seen;       // gathered by this call
    std::vector<uint16_t*> bound;    // ... into this output
    try {
        seen.assign(static_cast<size_t>(n_sub), 0);
        bound.assign(static_cast<size_t>(n_sub), nullptr);
        for (int32_t i = 0; i < n; ++i) {
            const int32_t k = ks[i];
            if (p->status[k] != ZERO3_NOT_AVAILABLE || seen[k]) {
                // a later fetch adds a reference and must name the same out
                const uint16_t* want = seen[k] ? bound[k] : p->fetched_out[k];
                if (outs[i] != want) return ZERO3_ESTATE;
                continue;
            }
            zero3_status st = z3::check_gather_sources(p, k, sparam, persist_param, outs[i]);
            if (st != ZERO3_OK) return st;
            seen[k] = 1;
            bound[k] = outs[i];
            gather.push_back(k);
            gather_out.push_back(outs[i]);
        }
    } catch (const std::bad_alloc&) {
        return ZERO3_ENOMEM;
    }
    for (int32_t k : gather) {
        if (!p->events[k] &&
            cudaEventCreateWithFlags(&p->events[k], cudaEventDisableTiming) != cudaSuccess) {
            p->events[k] = nullptr;
            return ZERO3_ECUDA;
        }
    }
    zero3_status st = z3::gather_submodules(p, gather.data(), static_cast<int64_t>(gather.size()),
                                            sparam, persist_param, gather_out.data(), stream);
    if (st != ZERO3_OK) return st;
    // every event first: a failed call leaves every status and count as it was
    for (int32_t k : gather)
        if (cudaEventRecord(p->events[k], stream) != cudaSuccess) return ZERO3_ECUDA;
    for (size_t j = 0; j < gather.size(); ++j) {
        const int32_t k = gather[j];
        p->status[k] = ZERO3_INFLIGHT;
        p->refs[k] = 0;
        p->fetched_out[k] = gather_out[j];
    }
    for (int32_t i = 0; i < n; ++i) p->refs[ks[i]] += 1;
    return ZERO3_OK;
}

zero3_status zero3_release_submodule(zero3_plan* p, int32_t k) {
    if (!p || k < 0 || k >= static_cast<int32_t>(p->sub_tensors.size())) return ZERO3_EINVAL;
    if (p->status[k] == ZERO3_NOT_AVAILABLE) return ZERO3_ESTATE;
    p->refs[k] -= 1;
    if (p->refs[k] == 0) {
        p->status[k] = ZERO3_NOT_AVAILABLE;
        p->fetched_out[k] = nullptr;
    }
    return ZERO3_OK;
}

zero3_status zero3_submodule_status(zero3_plan* p, int32_t k, int32_t* status) {
    if (!p || !status || k < 0 || k >= static_cast<int32_t>(p->sub_tensors.size()))
        return ZERO3_EINVAL;
    if (p->status[k] == ZERO3_INFLIGHT) {
        const cudaError_t e = cudaEventQuery(p->events[k]);
        if (e == cudaSuccess)
            p->status[k] = ZERO3_AVAILABLE;
        else if (e != cudaErrorNotReady)
            return ZERO3_ECUDA;
    }
    *status = p->status[k];
    return ZERO3_OK;
}

zero3_status zero3_submodule_wait(zero3_plan* p, int32_t k) {
    if (!p || k < 0 || k >= static_cast<int32_t>(p->sub_tensors.size())) return ZERO3_EINVAL;
    if (p->status[k] == ZERO3_NOT_AVAILABLE) return ZERO3_ESTATE;
    if (p->status[k] == ZERO3_INFLIGHT) {
        if (cudaEventSynchronize(p->events[k]) != cudaSuccess) return ZERO3_ECUDA;
        p->status[k] = ZERO3_AVAILABLE;
    }
    return ZERO3_OK;
}

zero3_status zero3_sync(zero3_stream stream) {
    return cuda_status(cudaStreamSynchronize(stream));
}

}  // extern "C"
