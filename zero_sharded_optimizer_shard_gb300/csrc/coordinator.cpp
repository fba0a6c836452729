// Prefetching submodule coordinator.
//
// Before a submodule runs, its parameters must be gathered from the shards;
// to hide that, the gathers of the submodules that come next are issued while
// the current one still computes ("DeepSpeed Zero-3 的参数分区与按需访问机制",
// hotelren.com: fetch_sub_module starts collecting later layers' parameters
// before the current layer has finished; the ZeroParamStatus state machine
// NOT_AVAILABLE -> INFLIGHT -> AVAILABLE -> NOT_AVAILABLE).  The knobs follow
// the pages' stage-3 settings (ZERO tutorial, cnhsyj.com, section 3.2;
// hotelren, tuning list): stage3_prefetch_bucket_size bounds the elements
// gathered ahead of use, stage3_max_live_parameters bounds the gathered
// elements held at once, stage3_max_reuse_distance keeps a released
// submodule gathered when it is needed again soon.
//
// Design on one GPU:
//  * Gathers run on `prefetch_stream`; consumers run on `compute_stream`,
//    which waits on the submodule's ready event before its first use.
//  * Gathered copies live in a caller-provided arena; a host-side first-fit
//    allocator hands out ranges.  A freed range may hold data a consumer on
//    the compute stream has not read yet, so each release records an event
//    on the compute stream and a later gather into that range first makes
//    the prefetch stream wait on it.  Events on one stream complete in
//    order, so a ring of release events suffices: waiting on a later event of
//    the ring implies the earlier ones.
//  * The fetch order comes from a trace given at creation, or recorded during
//    the first step (no prefetch in that step).  A fetch that departs from the
//    trace disables prefetching until the next step.
//  * At a step boundary (after the optimizer step was enqueued on the compute
//    stream) every gathered copy is stale: all are dropped, and the prefetch
//    stream waits for the optimizer step before gathering again.
//  * Prefetches are issued as batches: every submodule that fits the budgets
//    is placed in the arena first, the prefetch stream waits once for the
//    latest release among their ranges, and one zero3_fetch_submodules-style
//    gather (a few launches of up to 512 pieces) fills them all ("allgather
//    bucket": many small gathers aggregated into few large ones, ZERO
//    tutorial, cnhsyj.com, section 3.1).  Each submodule's ready event is
//    recorded after the batch; events on the prefetch stream complete in
//    order, so the compute stream waits on a ready event only if it has not
//    already waited on a later one.
#include <algorithm>
#include <new>
#include <vector>

#include "internal.h"

namespace {

constexpr int kReleaseRing = 64;

struct FreeRange {
    int64_t off, len;
    uint64_t seq;  // release event that freed it (0: never used)
};

}  // namespace

struct zero3_coordinator {
    zero3_plan* plan = nullptr;
    std::vector<const uint16_t*> sparam;
    const uint16_t* persist = nullptr;
    uint16_t* arena = nullptr;
    int64_t arena_elems = 0;
    zero3_prefetch_config cfg{};
    cudaStream_t compute = nullptr, prefetch = nullptr;

    std::vector<int32_t> trace;      // expected fetch order of one step
    std::vector<int32_t> recording;  // order seen in the current step
    bool trace_ok = false;
    int64_t pos = 0;                 // next trace position
    // Index of the trace, rebuilt whenever it is set: the positions at which
    // each submodule is fetched (ascending), and prefix sums of the fetched
    // elements, so next use and reuse distance cost O(log) and O(1).
    std::vector<std::vector<int64_t>> uses;
    std::vector<int64_t> prefix;

    int32_t n_sub = 0;
    std::vector<int32_t> status, refs;
    std::vector<int64_t> off;        // arena offset of a live submodule, -1 otherwise
    std::vector<uint8_t> ahead;      // gathered ahead of use and not fetched yet
    std::vector<cudaEvent_t> ready;
    std::vector<uint64_t> ready_seq;  // position of ready[k] on the prefetch stream
    uint64_t prefetch_seq = 0;        // events recorded on the prefetch stream so far
    uint64_t compute_waited = 0;      // latest prefetch position the compute stream waited on
    int64_t live = 0, ahead_elems = 0;

    std::vector<FreeRange> free_list;
    cudaEvent_t rel[kReleaseRing] = {};
    uint64_t rel_seq = 0;
    cudaEvent_t step_event = nullptr;

    zero3_coordinator_stats stats{};

    ~zero3_coordinator() {
        for (cudaEvent_t e : ready)
            if (e) cudaEventDestroy(e);
        for (cudaEvent_t e : rel)
            if (e) cudaEventDestroy(e);
        if (step_event) cudaEventDestroy(step_event);
    }
};

namespace {

int64_t numel_of(const zero3_coordinator* c, int32_t k) { return c->plan->sub_numel[k]; }

// Arena ranges are whole multiples of 8 elements (16 bytes), so every
// gathered copy starts 16-byte aligned like the arena itself: the gather
// kernel's vector path stores 16 bytes at a time relative to that start.
int64_t span_of(const zero3_coordinator* c, int32_t k) { return (numel_of(c, k) + 7) / 8 * 8; }

void free_insert(zero3_coordinator* c, int64_t off, int64_t len, uint64_t seq) {
    if (len <= 0) return;
    auto& fl = c->free_list;
    auto it = std::lower_bound(fl.begin(), fl.end(), off,
                               [](const FreeRange& r, int64_t o) { return r.off < o; });
    it = fl.insert(it, FreeRange{off, len, seq});
    // merge with neighbours; a merged range carries the latest release
    size_t i = static_cast<size_t>(it - fl.begin());
    if (i + 1 < fl.size() && fl[i].off + fl[i].len == fl[i + 1].off) {
        fl[i].len += fl[i + 1].len;
        fl[i].seq = std::max(fl[i].seq, fl[i + 1].seq);
        fl.erase(fl.begin() + static_cast<long>(i) + 1);
    }
    if (i > 0 && fl[i - 1].off + fl[i - 1].len == fl[i].off) {
        fl[i - 1].len += fl[i].len;
        fl[i - 1].seq = std::max(fl[i - 1].seq, fl[i].seq);
        fl.erase(fl.begin() + static_cast<long>(i));
    }
}

// First fit.  Returns the offset (or -1) and the release the range waits on.
int64_t free_take(zero3_coordinator* c, int64_t len, uint64_t* seq) {
    auto& fl = c->free_list;
    for (size_t i = 0; i < fl.size(); ++i) {
        if (fl[i].len >= len) {
            const int64_t o = fl[i].off;
            *seq = fl[i].seq;
            fl[i].off += len;
            fl[i].len -= len;
            if (fl[i].len == 0) fl.erase(fl.begin() + static_cast<long>(i));
            return o;
        }
    }
    return -1;
}

// Records a release point on the compute stream; returns its sequence number.
zero3_status record_release(zero3_coordinator* c, uint64_t* seq) {
    const uint64_t s = ++c->rel_seq;
    if (cudaEventRecord(c->rel[s % kReleaseRing], c->compute) != cudaSuccess) return ZERO3_ECUDA;
    *seq = s;
    return ZERO3_OK;
}

zero3_status drop(zero3_coordinator* c, int32_t k) {
    uint64_t seq = 0;
    zero3_status st = record_release(c, &seq);
    if (st != ZERO3_OK) return st;
    free_insert(c, c->off[k], span_of(c, k), seq);
    c->live -= numel_of(c, k);
    if (c->ahead[k]) c->ahead_elems -= numel_of(c, k);
    c->ahead[k] = 0;
    c->off[k] = -1;
    c->status[k] = ZERO3_NOT_AVAILABLE;
    return ZERO3_OK;
}

// Rebuilds the index of the trace (may throw std::bad_alloc).
void index_trace(zero3_coordinator* c) {
    c->uses.assign(static_cast<size_t>(c->n_sub), {});
    c->prefix.assign(c->trace.size() + 1, 0);
    for (size_t j = 0; j < c->trace.size(); ++j) {
        c->uses[static_cast<size_t>(c->trace[j])].push_back(static_cast<int64_t>(j));
        c->prefix[j + 1] = c->prefix[j] + numel_of(c, c->trace[j]);
    }
}

// Next trace position >= from at which k is fetched again, or -1.
int64_t next_use(const zero3_coordinator* c, int32_t k, int64_t from) {
    if (!c->trace_ok) return -1;
    const std::vector<int64_t>& u = c->uses[static_cast<size_t>(k)];
    const auto it = std::lower_bound(u.begin(), u.end(), from);
    return it == u.end() ? -1 : *it;
}

// Gathered elements fetched between trace positions [from, to).
int64_t distance(const zero3_coordinator* c, int64_t from, int64_t to) {
    return c->prefix[static_cast<size_t>(to)] - c->prefix[static_cast<size_t>(from)];
}

// Gathers submodule k into a new arena range on the prefetch stream.  With
// `evict`, unreferenced kept copies are dropped (farthest next use first)
// when the arena or the live budget is exhausted.  Returns ZERO3_ENOMEM when
// there is no room.
zero3_status gather(zero3_coordinator* c, int32_t k, bool evict) {
    const int64_t n = numel_of(c, k);
    if (n == 0) {  // nothing to gather: an empty view at the arena's start
        if (cudaEventRecord(c->ready[k], c->prefetch) != cudaSuccess) return ZERO3_ECUDA;
        c->ready_seq[k] = ++c->prefetch_seq;
        c->off[k] = 0;
        c->status[k] = ZERO3_INFLIGHT;
        return ZERO3_OK;
    }
    for (;;) {
        uint64_t seq = 0;
        const bool budget = c->live + n <= c->cfg.max_live_parameters;
        const int64_t o = budget ? free_take(c, span_of(c, k), &seq) : -1;
        if (o >= 0) {
            if (seq > 0 &&
                cudaStreamWaitEvent(c->prefetch, c->rel[seq % kReleaseRing], 0) != cudaSuccess)
                return ZERO3_ECUDA;
            uint16_t* outs[1] = {c->arena + o};
            int64_t launches = 0;
            zero3_status st = z3::gather_submodules(c->plan, &k, 1, c->sparam.data(), c->persist,
                                                    outs, c->prefetch, &launches);
            if (st != ZERO3_OK) return st;
            if (cudaEventRecord(c->ready[k], c->prefetch) != cudaSuccess) return ZERO3_ECUDA;
            c->ready_seq[k] = ++c->prefetch_seq;
            c->off[k] = o;
            c->live += n;
            c->status[k] = ZERO3_INFLIGHT;
            c->stats.gathers += 1;
            c->stats.gather_calls += 1;
            c->stats.gather_launches += launches;
            c->stats.gathered_elems += n;
            if (c->live > c->stats.peak_live_elems) c->stats.peak_live_elems = c->live;
            return ZERO3_OK;
        }
        if (!evict) return ZERO3_ENOMEM;
        // drop the unreferenced copy (kept, or gathered ahead and not used
        // yet) whose next use is farthest away
        int32_t victim = -1;
        int64_t far = -2;
        for (int32_t j = 0; j < c->n_sub; ++j) {
            if (j == k || c->off[j] < 0 || c->refs[j] > 0) continue;
            int64_t u = next_use(c, j, c->pos);
            if (u < 0) u = INT64_MAX;
            if (u > far) {
                far = u;
                victim = j;
            }
        }
        if (victim < 0) return ZERO3_ENOMEM;
        zero3_status st = drop(c, victim);
        if (st != ZERO3_OK) return st;
        c->stats.evictions += 1;
    }
}

// Issues gathers for the trace entries after the current position while the
// prefetch budget and the live budget allow, as one batch: arena ranges for
// every submodule first, one wait for the latest release among them, one
// gather of all of them, then their ready events.
zero3_status prefetch_ahead(zero3_coordinator* c) {
    if (!c->trace_ok || c->cfg.prefetch_bucket_size <= 0) return ZERO3_OK;
    std::vector<int32_t> ks;
    std::vector<uint16_t*> outs;
    std::vector<uint64_t> seqs;  // the release each taken range waits for
    uint64_t wait_seq = 0;
    const size_t most = c->trace.size() - static_cast<size_t>(c->pos);
    try {  // no allocation after this: the loop below cannot throw
        ks.reserve(most);
        outs.reserve(most);
        seqs.reserve(most);
    } catch (const std::bad_alloc&) {
        return ZERO3_ENOMEM;
    }
    {
        for (int64_t j = c->pos; j < static_cast<int64_t>(c->trace.size()); ++j) {
            const int32_t k = c->trace[j];
            if (c->off[k] >= 0) continue;  // already gathered (ahead, kept, or in this batch)
            const int64_t n = numel_of(c, k);
            if (c->ahead_elems + n > c->cfg.prefetch_bucket_size) break;
            if (c->live + n > c->cfg.max_live_parameters) break;
            int64_t o = 0;
            uint64_t seq = 0;
            if (n > 0) {
                o = free_take(c, span_of(c, k), &seq);
                if (o < 0) break;  // no room now: try again at the next fetch
                wait_seq = std::max(wait_seq, seq);
            }
            ks.push_back(k);
            outs.push_back(c->arena + o);
            seqs.push_back(seq);
            c->off[k] = o;
            c->live += n;
            c->status[k] = ZERO3_INFLIGHT;
            c->ahead[k] = 1;
            c->ahead_elems += n;
        }
    }
    if (ks.empty()) return ZERO3_OK;
    // a batch that cannot be issued leaves nothing behind: its ranges return
    // to the free list and its submodules to NOT_AVAILABLE
    auto undo = [c, &ks, &seqs]() {
        for (size_t i = 0; i < ks.size(); ++i) {
            const int32_t k = ks[i];
            const int64_t n = numel_of(c, k);
            if (n > 0) free_insert(c, c->off[k], span_of(c, k), seqs[i]);
            c->live -= n;
            c->ahead_elems -= n;
            c->ahead[k] = 0;
            c->off[k] = -1;
            c->status[k] = ZERO3_NOT_AVAILABLE;
        }
    };
    // release events of one stream complete in order: the latest covers all
    if (wait_seq > 0 &&
        cudaStreamWaitEvent(c->prefetch, c->rel[wait_seq % kReleaseRing], 0) != cudaSuccess) {
        undo();
        return ZERO3_ECUDA;
    }
    int64_t launches = 0;
    zero3_status st = z3::gather_submodules(c->plan, ks.data(), static_cast<int64_t>(ks.size()),
                                            c->sparam.data(), c->persist, outs.data(), c->prefetch,
                                            &launches);
    if (st != ZERO3_OK) {
        undo();
        return st;
    }
    const uint64_t seq = ++c->prefetch_seq;  // every event below marks this position
    for (int32_t k : ks) {
        if (cudaEventRecord(c->ready[k], c->prefetch) != cudaSuccess) return ZERO3_ECUDA;
        c->ready_seq[k] = seq;
        const int64_t n = numel_of(c, k);
        c->stats.prefetched += 1;
        if (n > 0) {  // an empty submodule is a view, not a gather
            c->stats.gathers += 1;
            c->stats.gathered_elems += n;
        }
    }
    if (c->live > c->stats.peak_live_elems) c->stats.peak_live_elems = c->live;
    c->stats.gather_calls += 1;
    c->stats.gather_launches += launches;
    return ZERO3_OK;
}

bool valid_k(const zero3_coordinator* c, int32_t k) { return k >= 0 && k < c->n_sub; }

}  // namespace

extern "C" {

zero3_status zero3_coordinator_create(zero3_plan* plan, const int32_t* trace, int64_t n_trace,
                                      const uint16_t* const* sparam,
                                      const uint16_t* persist_param, uint16_t* arena,
                                      int64_t arena_elems, const zero3_prefetch_config* cfg,
                                      zero3_stream compute_stream, zero3_stream prefetch_stream,
                                      zero3_coordinator** out) {
    if (!out) return ZERO3_EINVAL;
    *out = nullptr;
    if (!plan || !cfg || n_trace < 0 || (n_trace > 0 && !trace) || arena_elems < 0) return ZERO3_EINVAL;
    if (cfg->prefetch_bucket_size < 0 || cfg->max_live_parameters < 0 ||
        cfg->max_reuse_distance < 0)
        return ZERO3_EINVAL;
    if (compute_stream == prefetch_stream) return ZERO3_EINVAL;
    if (arena_elems > 0 && (!arena || (reinterpret_cast<uintptr_t>(arena) & 15u)))
        return ZERO3_EINVAL;
    const int32_t n_sub = static_cast<int32_t>(plan->sub_tensors.size());
    int64_t biggest = 0;
    for (int32_t k = 0; k < n_sub; ++k) biggest = std::max(biggest, plan->sub_numel[k]);
    const int64_t biggest_span = (biggest + 7) / 8 * 8;
    // the sources of every submodule, checked once
    for (int64_t t = 0; t < static_cast<int64_t>(plan->numel.size()); ++t) {
        if (plan->numel[t] == 0) continue;
        if (plan->persistent[t]) {
            if (!persist_param || (reinterpret_cast<uintptr_t>(persist_param) & 15u))
                return ZERO3_EINVAL;
        } else {
            if (!sparam) return ZERO3_EINVAL;
            for (int64_t s = plan->seg_begin[t]; s < plan->seg_begin[t + 1]; ++s) {
                const uint16_t* src = sparam[plan->segs[s].rank];
                if (!src || (reinterpret_cast<uintptr_t>(src) & 15u)) return ZERO3_EINVAL;
            }
        }
    }
    if (biggest_span > arena_elems || biggest > cfg->max_live_parameters) return ZERO3_EINVAL;
    for (int64_t j = 0; j < n_trace; ++j)
        if (trace[j] < 0 || trace[j] >= n_sub) return ZERO3_EINVAL;

    zero3_coordinator* c = new (std::nothrow) zero3_coordinator;
    if (!c) return ZERO3_ENOMEM;
    try {
        c->plan = plan;
        c->sparam.assign(plan->n_ranks, nullptr);
        if (sparam)
            for (int r = 0; r < plan->n_ranks; ++r) c->sparam[r] = sparam[r];
        c->persist = persist_param;
        c->arena = arena;
        c->arena_elems = arena_elems;
        c->cfg = *cfg;
        c->compute = compute_stream;
        c->prefetch = prefetch_stream;
        c->trace.assign(trace, trace + n_trace);
        c->trace_ok = n_trace > 0;
        c->n_sub = n_sub;
        index_trace(c);
        c->status.assign(n_sub, ZERO3_NOT_AVAILABLE);
        c->refs.assign(n_sub, 0);
        c->off.assign(n_sub, -1);
        c->ahead.assign(n_sub, 0);
        c->ready.assign(n_sub, nullptr);
        c->ready_seq.assign(n_sub, 0);
        // only whole 8-element units of the arena are handed out.  Free
        // ranges are separated by live ones, so there are at most n_sub + 1
        // of them: with that capacity reserved, inserting never allocates
        // (and never throws) later.
        c->free_list.reserve(static_cast<size_t>(n_sub) + 2);
        if (arena_elems >= 8) c->free_list.push_back(FreeRange{0, arena_elems / 8 * 8, 0});
    } catch (const std::bad_alloc&) {
        delete c;
        return ZERO3_ENOMEM;
    }
    bool ok = true;
    for (int32_t k = 0; k < n_sub && ok; ++k)
        ok = cudaEventCreateWithFlags(&c->ready[k], cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < kReleaseRing && ok; ++i)
        ok = cudaEventCreateWithFlags(&c->rel[i], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&c->step_event, cudaEventDisableTiming) == cudaSuccess;
    // the first gathers read shards written by work already queued on the
    // compute stream (initialisation, a previous optimizer step)
    ok = ok && cudaEventRecord(c->step_event, compute_stream) == cudaSuccess &&
         cudaStreamWaitEvent(prefetch_stream, c->step_event, 0) == cudaSuccess;
    if (!ok) {
        delete c;
        return ZERO3_ECUDA;
    }
    *out = c;
    return ZERO3_OK;
}

zero3_status zero3_coordinator_fetch(zero3_coordinator* c, int32_t k, uint16_t** out) {
    if (!c || !out || !valid_k(c, k)) return ZERO3_EINVAL;
    // follow the trace; a departure disables prefetching until the next step
    if (c->trace_ok) {
        if (c->pos < static_cast<int64_t>(c->trace.size()) && c->trace[c->pos] == k) {
            c->pos += 1;
        } else {
            c->trace_ok = false;
            c->stats.trace_misses += 1;
        }
    }
    try {
        c->recording.push_back(k);
    } catch (const std::bad_alloc&) {
        return ZERO3_ENOMEM;
    }
    if (c->off[k] < 0) {
        zero3_status st = gather(c, k, true);
        if (st != ZERO3_OK) return st;
    } else if (c->ahead[k]) {
        c->stats.prefetch_hits += 1;
    } else if (c->refs[k] == 0) {
        c->stats.reuse_hits += 1;
    }
    if (c->ahead[k]) {
        c->ahead[k] = 0;
        c->ahead_elems -= numel_of(c, k);
    }
    // skip a wait that an earlier wait on a later prefetch event implies
    if (c->ready_seq[k] > c->compute_waited) {
        if (cudaStreamWaitEvent(c->compute, c->ready[k], 0) != cudaSuccess) return ZERO3_ECUDA;
        c->compute_waited = c->ready_seq[k];
        c->stats.compute_waits += 1;
    }
    c->refs[k] += 1;
    zero3_status st = prefetch_ahead(c);
    if (st != ZERO3_OK) return st;
    *out = c->arena + c->off[k];
    return ZERO3_OK;
}

zero3_status zero3_coordinator_release(zero3_coordinator* c, int32_t k) {
    if (!c || !valid_k(c, k)) return ZERO3_EINVAL;
    if (c->off[k] < 0 || c->refs[k] == 0) return ZERO3_ESTATE;
    c->refs[k] -= 1;
    if (c->refs[k] > 0) return ZERO3_OK;
    // keep it gathered when it is needed again within the reuse distance
    const int64_t u = next_use(c, k, c->pos);
    if (u >= 0 && distance(c, c->pos, u) <= c->cfg.max_reuse_distance) return ZERO3_OK;
    return drop(c, k);
}

zero3_status zero3_coordinator_status(zero3_coordinator* c, int32_t k, int32_t* status) {
    if (!c || !status || !valid_k(c, k)) return ZERO3_EINVAL;
    if (c->status[k] == ZERO3_INFLIGHT) {
        const cudaError_t e = cudaEventQuery(c->ready[k]);
        if (e == cudaSuccess)
            c->status[k] = ZERO3_AVAILABLE;
        else if (e != cudaErrorNotReady)
            return ZERO3_ECUDA;
    }
    *status = c->status[k];
    return ZERO3_OK;
}

zero3_status zero3_coordinator_next_step(zero3_coordinator* c) {
    if (!c) return ZERO3_EINVAL;
    for (int32_t k = 0; k < c->n_sub; ++k)
        if (c->refs[k] > 0) return ZERO3_ESTATE;
    // every gathered copy predates the optimizer step: drop them all
    for (int32_t k = 0; k < c->n_sub; ++k) {
        if (c->off[k] >= 0) {
            zero3_status st = drop(c, k);
            if (st != ZERO3_OK) return st;
        }
    }
    // gathers of the next step read the updated shards
    if (cudaEventRecord(c->step_event, c->compute) != cudaSuccess ||
        cudaStreamWaitEvent(c->prefetch, c->step_event, 0) != cudaSuccess)
        return ZERO3_ECUDA;
    if (!c->trace_ok || c->trace.empty()) {
        // adopt the order seen in this step
        c->trace.swap(c->recording);
        c->trace_ok = !c->trace.empty();
        try {
            index_trace(c);
        } catch (const std::bad_alloc&) {
            c->trace_ok = false;
            return ZERO3_ENOMEM;
        }
    }
    c->recording.clear();
    c->pos = 0;
    c->stats.steps += 1;
    return prefetch_ahead(c);
}

zero3_status zero3_coordinator_get_stats(const zero3_coordinator* c,
                                         zero3_coordinator_stats* stats) {
    if (!c || !stats) return ZERO3_EINVAL;
    *stats = c->stats;
    stats->live_elems = c->live;
    return ZERO3_OK;
}

void zero3_coordinator_destroy(zero3_coordinator* c) { delete c; }

}  // extern "C"
