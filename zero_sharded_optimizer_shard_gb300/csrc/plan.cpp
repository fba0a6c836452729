// Host planner: flatten, classify, pad and shard a parameter list; the
// per-step AdamW scalars; the model-state and communication accounting.
//
// Partition rules ("DeepSpeed Zero-3 的参数分区与按需访问机制", hotelren.com,
// 小参数驻留; ZERO tutorial, cnhsyj.com, sections 2.1 and 3.2;
// "ddp-to-zero-memory-sharding", 111qqz.com, section
// "ZeRO-3：参数为什么也可以分片"): tensors below the persistence threshold
// stay whole on every rank; the others are concatenated in list order,
// zero-padded to a multiple of N_d and cut into N_d contiguous shards.
#include <cmath>
#include <new>

#include "internal.h"

namespace z3 {

Scalars make_scalars(const zero3_adamw_hparams& hp, int64_t t, int32_t n_ranks) {
    // Powers by repeated products, everything in double, rounded once to
    // binary32 (AdamW with Kingma & Ba bias correction; decoupled decay).
    // A per-thread cache of the last (beta1, beta2, t) makes consecutive
    // steps cost one product each; the products are the same sequence as a
    // recomputation from t = 0.
    thread_local double c_beta1 = -1.0, c_beta2 = -1.0, c_b1t = 1.0, c_b2t = 1.0;
    thread_local int64_t c_t = -1;
    double b1t = 1.0, b2t = 1.0;
    int64_t k0 = 0;
    if (c_beta1 == hp.beta1 && c_beta2 == hp.beta2 && c_t >= 0 && c_t <= t) {
        b1t = c_b1t;
        b2t = c_b2t;
        k0 = c_t;
    }
    for (int64_t k = k0; k < t; ++k) {
        b1t *= hp.beta1;
        b2t *= hp.beta2;
    }
    c_beta1 = hp.beta1;
    c_beta2 = hp.beta2;
    c_b1t = b1t;
    c_b2t = b2t;
    c_t = t;
    const double bc1 = 1.0 - b1t;
    const double bc2 = 1.0 - b2t;
    Scalars s;
    s.step_size = static_cast<float>(hp.lr / bc1);
    s.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
    s.decay = static_cast<float>(1.0 - hp.lr * hp.weight_decay);
    s.b1 = static_cast<float>(hp.beta1);
    s.omb1 = static_cast<float>(1.0 - hp.beta1);
    s.b2 = static_cast<float>(hp.beta2);
    s.omb2 = static_cast<float>(1.0 - hp.beta2);
    s.eps = static_cast<float>(hp.eps);
    s.inv_nd = static_cast<float>(1.0 / static_cast<double>(n_ranks));
    return s;
}

}  // namespace z3

extern "C" {

zero3_status zero3_partition(const int64_t* numels, const int32_t* submodule_of, int64_t n_tensors,
                             int32_t n_ranks, int64_t persistence_threshold,
                             int64_t reduce_bucket_size, zero3_plan** out) {
    if (!out) return ZERO3_EINVAL;
    *out = nullptr;
    if (n_tensors < 0 || (n_tensors > 0 && !numels)) return ZERO3_EINVAL;
    if (n_ranks < 1 || n_ranks > ZERO3_MAX_RANKS) return ZERO3_EINVAL;
    if (persistence_threshold < 0 || reduce_bucket_size < 1) return ZERO3_EINVAL;
    for (int64_t t = 0; t < n_tensors; ++t) {
        if (numels[t] < 0) return ZERO3_EINVAL;
        if (submodule_of && submodule_of[t] < 0) return ZERO3_EINVAL;
    }
    if (!submodule_of && n_tensors > INT32_MAX) return ZERO3_EINVAL;

    zero3_plan* p = new (std::nothrow) zero3_plan;
    if (!p) return ZERO3_ENOMEM;
    try {
        p->n_ranks = n_ranks;
        p->threshold = persistence_threshold;
        p->bucket = reduce_bucket_size;
        p->numel.assign(numels, numels + n_tensors);
        p->submodule.resize(n_tensors);
        p->persistent.resize(n_tensors);
        p->offset.resize(n_tensors);
        int64_t flat = 0, pers = 0;
        int32_t n_sub = 0;
        for (int64_t t = 0; t < n_tensors; ++t) {
            p->submodule[t] = submodule_of ? submodule_of[t] : static_cast<int32_t>(t);
            if (p->submodule[t] + 1 > n_sub) n_sub = p->submodule[t] + 1;
            const bool pers_t = numels[t] < persistence_threshold;
            p->persistent[t] = pers_t ? 1 : 0;
            if (pers_t) {
                p->offset[t] = pers;
                pers += numels[t];
            } else {
                p->offset[t] = flat;
                flat += numels[t];
                p->n_partitioned++;
            }
        }
        p->psi_p = flat;
        p->psi_s = pers;
        p->psi_pad = (flat + n_ranks - 1) / n_ranks * n_ranks;
        p->S = p->psi_pad / n_ranks;
        // segments: split [off, off+numel) at multiples of S
        p->seg_begin.resize(n_tensors + 1);
        for (int64_t t = 0; t < n_tensors; ++t) {
            p->seg_begin[t] = static_cast<int64_t>(p->segs.size());
            if (p->persistent[t]) continue;
            int64_t f = p->offset[t];
            const int64_t end = f + numels[t];
            while (f < end) {
                const int64_t r = f / p->S;
                int64_t stop = (r + 1) * p->S;
                if (stop > end) stop = end;
                zero3_segment s;
                s.rank = static_cast<int32_t>(r);
                s.reserved = 0;
                s.shard_off = f - r * p->S;
                s.tensor_off = f - p->offset[t];
                s.len = stop - f;
                p->segs.push_back(s);
                f = stop;
            }
        }
        p->seg_begin[n_tensors] = static_cast<int64_t>(p->segs.size());
        p->sub_tensors.resize(n_sub);
        p->sub_numel.assign(n_sub, 0);
        for (int64_t t = 0; t < n_tensors; ++t) {
            p->sub_tensors[p->submodule[t]].push_back(t);
            p->sub_numel[p->submodule[t]] += numels[t];
        }
        p->status.assign(n_sub, ZERO3_NOT_AVAILABLE);
        p->refs.assign(n_sub, 0);
        p->fetched_out.assign(n_sub, nullptr);
        p->events.assign(n_sub, nullptr);
    } catch (const std::bad_alloc&) {
        delete p;
        return ZERO3_ENOMEM;
    }
    *out = p;
    return ZERO3_OK;
}

zero3_status zero3_plan_info_get(const zero3_plan* p, zero3_plan_info* info) {
    if (!p || !info) return ZERO3_EINVAL;
    info->n_ranks = p->n_ranks;
    info->n_submodules = static_cast<int32_t>(p->sub_tensors.size());
    info->n_tensors = static_cast<int64_t>(p->numel.size());
    info->n_partitioned = p->n_partitioned;
    info->n_persistent = info->n_tensors - p->n_partitioned;
    info->psi_p = p->psi_p;
    info->psi_pad = p->psi_pad;
    info->shard_len = p->S;
    info->psi_s = p->psi_s;
    info->persistence_threshold = p->threshold;
    info->reduce_bucket_size = p->bucket;
    info->n_buckets = (p->psi_pad + p->bucket - 1) / p->bucket;
    return ZERO3_OK;
}

zero3_status zero3_plan_tensor(const zero3_plan* p, int64_t t, zero3_tensor_info* info) {
    if (!p || !info || t < 0 || t >= static_cast<int64_t>(p->numel.size())) return ZERO3_EINVAL;
    info->numel = p->numel[t];
    info->offset = p->offset[t];
    info->persistent = p->persistent[t];
    info->submodule = p->submodule[t];
    const int64_t b = p->seg_begin[t], e = p->seg_begin[t + 1];
    info->n_segments = e - b;
    info->first_rank = (e > b) ? p->segs[b].rank : -1;
    info->last_rank = (e > b) ? p->segs[e - 1].rank : -1;
    return ZERO3_OK;
}

zero3_status zero3_plan_segments(const zero3_plan* p, int64_t t, zero3_segment* out, int64_t cap,
                                 int64_t* n) {
    if (!p || !n || t < 0 || t >= static_cast<int64_t>(p->numel.size()) || cap < 0)
        return ZERO3_EINVAL;
    if (cap > 0 && !out) return ZERO3_EINVAL;
    const int64_t b = p->seg_begin[t], e = p->seg_begin[t + 1];
    *n = e - b;
    for (int64_t k = 0; k < e - b && k < cap; ++k) out[k] = p->segs[b + k];
    return ZERO3_OK;
}

zero3_status zero3_plan_bucket(const zero3_plan* p, int64_t b, int64_t* lo, int64_t* hi) {
    if (!p || !lo || !hi) return ZERO3_EINVAL;
    const int64_t nb = (p->psi_pad + p->bucket - 1) / p->bucket;
    if (b < 0 || b >= nb) return ZERO3_EINVAL;
    *lo = b * p->bucket;
    *hi = (b + 1) * p->bucket < p->psi_pad ? (b + 1) * p->bucket : p->psi_pad;
    return ZERO3_OK;
}

zero3_status zero3_plan_submodule(const zero3_plan* p, int32_t k, int64_t* n_tensors,
                                  int64_t* numel) {
    if (!p || k < 0 || k >= static_cast<int32_t>(p->sub_tensors.size())) return ZERO3_EINVAL;
    if (n_tensors) *n_tensors = static_cast<int64_t>(p->sub_tensors[k].size());
    if (numel) *numel = p->sub_numel[k];
    return ZERO3_OK;
}

void zero3_plan_destroy(zero3_plan* p) {
    if (!p) return;
    for (cudaEvent_t e : p->events)
        if (e) cudaEventDestroy(e);
    delete p;
}

zero3_status zero3_memory_bytes(int32_t stage, double psi, int32_t n_d, double* bytes) {
    // (2+2+K)Ψ with K = 12 for Adam; the stage decides which terms are /N_d.
    if (!bytes || n_d < 1 || !(psi >= 0.0)) return ZERO3_EINVAL;
    const double K = 12.0, nd = static_cast<double>(n_d);
    switch (stage) {
        case 0: *bytes = (2.0 + 2.0 + K) * psi; break;
        case 1: *bytes = 2.0 * psi + 2.0 * psi + K * psi / nd; break;
        case 2: *bytes = 2.0 * psi + (2.0 + K) * psi / nd; break;
        case 3: *bytes = (2.0 + 2.0 + K) * psi / nd; break;
        default: return ZERO3_EINVAL;
    }
    return ZERO3_OK;
}

zero3_status zero3_plan_memory_bytes(const zero3_plan* p, int32_t stage, double* bytes) {
    // closed form on the padded partitioned elements + the persistent group,
    // which every rank keeps whole (2 + 2 + 12 bytes per element)
    if (!p || !bytes) return ZERO3_EINVAL;
    double part = 0.0;
    zero3_status st = zero3_memory_bytes(stage, static_cast<double>(p->psi_pad), p->n_ranks, &part);
    if (st != ZERO3_OK) return st;
    *bytes = part + 16.0 * static_cast<double>(p->psi_s);
    return ZERO3_OK;
}

zero3_status zero3_comm_elems(int32_t stage, double psi, int32_t n_d, double* elems) {
    // reduce-scatter + all-gather = 2Ψ; stage 3 gathers parameters twice.
    if (!elems || n_d < 1 || !(psi >= 0.0)) return ZERO3_EINVAL;
    double k;
    switch (stage) {
        case 0: case 1: case 2: k = 2.0; break;
        case 3: k = 3.0; break;
        default: return ZERO3_EINVAL;
    }
    const double nd = static_cast<double>(n_d);
    *elems = k * psi * (nd - 1.0) / nd;
    return ZERO3_OK;
}

const char* zero3_status_string(zero3_status s) {
    switch (s) {
        case ZERO3_OK: return "ok";
        case ZERO3_EINVAL: return "invalid argument";
        case ZERO3_ESTATE: return "invalid submodule state";
        case ZERO3_ECUDA: return "CUDA error";
        case ZERO3_ENOMEM: return "out of host memory";
        case ZERO3_EIO: return "checkpoint file error";
    }
    return "unknown status";
}

}  // extern "C"
