// Checkpoints of the sharded state and the consolidated 16-bit weights.
//
// Under ZeRO-3 each rank's state is a disjoint fragment, so checkpoints are
// saved per partition and restored by the same partitioning (ZERO tutorial,
// cnhsyj.com, section 4.3: save_checkpoint writes every partition,
// load_checkpoint restores them), or the weights are gathered into complete
// 16-bit tensors at save time ("DeepSpeed Zero-3 的参数分区与按需访问机制",
// stage3_gather_16bit_weights_on_model_save; encyclopedia entry
// "DeepSpeed ZeRO-3", section 应用: either gather full weights or save the
// shards and merge them later).
//
// File = header + raw little-endian arrays.  The header carries a fingerprint
// of the partition (rank count, threshold, element counts), so a shard can
// only be loaded into the partitioning that wrote it.
//
// Saves never write into the destination path directly: they write a
// temporary file beside it, flush it to disk and rename it over the path, so
// a failed or interrupted save (no space, a CUDA error mid-copy, a killed
// process) leaves the previous file as it was.  Loads check the header and
// the file's exact size before the first byte reaches device memory.
#include <sys/stat.h>
#include <unistd.h>

#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"

namespace {

constexpr char kMagic[8] = {'Z', 'E', 'R', 'O', '3', 'C', 'K', 'P'};
constexpr uint32_t kVersion = 1;
enum Kind : uint32_t { kShard = 1, kPersist = 2, kWeights16 = 3, kWeights32 = 4 };
constexpr int64_t kStage = int64_t(16) << 20;  // bytes per host staging chunk

struct Header {
    char magic[8];
    uint32_t version;
    uint32_t kind;
    int32_t rank;
    int32_t n_ranks;
    int64_t n_elems;
    int64_t t;
    uint64_t fingerprint;
};
static_assert(sizeof(Header) == 48, "checkpoint header layout");

// FNV-1a over the values that fix the partition.
uint64_t fingerprint(const zero3_plan* p) {
    uint64_t h = 14695981039346656037ull;  // FNV-1a 64 offset basis
    auto mix = [&h](int64_t x) {
        for (int k = 0; k < 8; ++k) {
            h ^= static_cast<uint64_t>((x >> (8 * k)) & 0xff);
            h *= 1099511628211ull;
        }
    };
    mix(p->n_ranks);
    mix(p->threshold);
    mix(static_cast<int64_t>(p->numel.size()));
    for (int64_t n : p->numel) mix(n);
    return h;
}

Header make_header(const zero3_plan* p, Kind kind, int32_t rank, int64_t n, int64_t t) {
    Header h;
    std::memcpy(h.magic, kMagic, 8);
    h.version = kVersion;
    h.kind = kind;
    h.rank = rank;
    h.n_ranks = p->n_ranks;
    h.n_elems = n;
    h.t = t;
    h.fingerprint = fingerprint(p);
    return h;
}

struct File {
    FILE* f = nullptr;
    File() = default;
    File(const File&) = delete;
    File& operator=(const File&) = delete;
    ~File() {
        if (f) std::fclose(f);
    }
};

// Output file written under a temporary name ("<path>.tmp.<pid>") and moved
// over `path` by commit(): fflush, fsync, fclose, rename.  Destroyed without
// a successful commit, it removes the temporary file and leaves `path`
// untouched.
struct AtomicFile {
    FILE* f = nullptr;
    std::string path, tmp;
    bool done = false;
    AtomicFile() = default;
    AtomicFile(const AtomicFile&) = delete;
    AtomicFile& operator=(const AtomicFile&) = delete;
    zero3_status open(const char* dst) {
        try {
            path = dst;
            tmp = path + ".tmp." + std::to_string(static_cast<long long>(getpid()));
        } catch (const std::bad_alloc&) {
            return ZERO3_ENOMEM;
        }
        f = std::fopen(tmp.c_str(), "wb");
        if (!f) {
            tmp.clear();
            return ZERO3_EIO;
        }
        return ZERO3_OK;
    }
    zero3_status commit() {
        const bool flushed = std::fflush(f) == 0 && fsync(fileno(f)) == 0;
        const bool closed = std::fclose(f) == 0;
        f = nullptr;
        if (!flushed || !closed || std::rename(tmp.c_str(), path.c_str()) != 0) return ZERO3_EIO;
        done = true;
        return ZERO3_OK;
    }
    ~AtomicFile() {
        if (f) std::fclose(f);
        if (!done && !tmp.empty()) std::remove(tmp.c_str());
    }
};

// Copies `bytes` of device memory at src to the file through a host buffer.
zero3_status write_device(FILE* f, const void* src, int64_t bytes, std::vector<char>& buf,
                          cudaStream_t s) {
    const char* p = static_cast<const char*>(src);
    for (int64_t off = 0; off < bytes; off += kStage) {
        const int64_t n = (bytes - off) < kStage ? (bytes - off) : kStage;
        if (cudaMemcpyAsync(buf.data(), p + off, n, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return ZERO3_ECUDA;
        if (std::fwrite(buf.data(), 1, n, f) != static_cast<size_t>(n)) return ZERO3_EIO;
    }
    return ZERO3_OK;
}

zero3_status read_device(FILE* f, void* dst, int64_t bytes, std::vector<char>& buf,
                         cudaStream_t s) {
    char* p = static_cast<char*>(dst);
    for (int64_t off = 0; off < bytes; off += kStage) {
        const int64_t n = (bytes - off) < kStage ? (bytes - off) : kStage;
        if (std::fread(buf.data(), 1, n, f) != static_cast<size_t>(n)) return ZERO3_EIO;
        if (cudaMemcpyAsync(p + off, buf.data(), n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return ZERO3_ECUDA;
    }
    return ZERO3_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Opens and validates a checkpoint file written for this plan: every header
// field, and a total size of exactly the header plus `payload` bytes (a
// truncated file or one with trailing bytes is rejected here, before any of
// it is read into device memory).
zero3_status open_checked(const zero3_plan* p, const char* path, Kind kind, int32_t rank,
                          int64_t n, int64_t payload, File& file, Header& h) {
    file.f = std::fopen(path, "rb");
    if (!file.f) return ZERO3_EIO;
    struct stat sb;
    if (fstat(fileno(file.f), &sb) != 0 ||
        static_cast<int64_t>(sb.st_size) != static_cast<int64_t>(sizeof(Header)) + payload)
        return ZERO3_EIO;
    if (std::fread(&h, sizeof(h), 1, file.f) != 1) return ZERO3_EIO;
    if (std::memcmp(h.magic, kMagic, 8) != 0 || h.version != kVersion || h.kind != kind ||
        h.rank != rank || h.n_ranks != p->n_ranks || h.n_elems != n ||
        h.fingerprint != fingerprint(p) || h.t < 0)
        return ZERO3_EIO;
    return ZERO3_OK;
}

zero3_status save_arrays(const zero3_plan* p, const char* path, Kind kind, int32_t rank,
                         int64_t n, int64_t t, const void* const* arrays, int n_arrays,
                         int elem_bytes, cudaStream_t s) {
    AtomicFile file;
    zero3_status st = file.open(path);
    if (st != ZERO3_OK) return st;
    const Header h = make_header(p, kind, rank, n, t);
    if (std::fwrite(&h, sizeof(h), 1, file.f) != 1) return ZERO3_EIO;
    std::vector<char> buf;
    try {
        buf.resize(kStage);
    } catch (const std::bad_alloc&) {
        return ZERO3_ENOMEM;
    }
    for (int k = 0; k < n_arrays; ++k) {
        st = write_device(file.f, arrays[k], n * elem_bytes, buf, s);
        if (st != ZERO3_OK) return st;
    }
    return file.commit();
}

zero3_status load_arrays(const zero3_plan* p, const char* path, Kind kind, int32_t rank,
                         int64_t n, int64_t* t, void* const* arrays, int n_arrays,
                         int elem_bytes, cudaStream_t s) {
    File file;
    Header h;
    zero3_status st =
        open_checked(p, path, kind, rank, n, n_arrays * n * elem_bytes, file, h);
    if (st != ZERO3_OK) return st;
    std::vector<char> buf;
    try {
        buf.resize(kStage);
    } catch (const std::bad_alloc&) {
        return ZERO3_ENOMEM;
    }
    for (int k = 0; k < n_arrays; ++k) {
        st = read_device(file.f, arrays[k], n * elem_bytes, buf, s);
        if (st != ZERO3_OK) return st;
    }
    *t = h.t;
    return ZERO3_OK;
}

// Copies `bytes` from file `in` at byte offset `off` to `out`.
zero3_status copy_range(FILE* in, int64_t off, int64_t bytes, FILE* out, std::vector<char>& buf) {
    if (std::fseek(in, static_cast<long>(off), SEEK_SET) != 0) return ZERO3_EIO;
    while (bytes > 0) {
        const int64_t n = bytes < static_cast<int64_t>(buf.size()) ? bytes
                                                                   : static_cast<int64_t>(buf.size());
        if (std::fread(buf.data(), 1, n, in) != static_cast<size_t>(n)) return ZERO3_EIO;
        if (std::fwrite(buf.data(), 1, n, out) != static_cast<size_t>(n)) return ZERO3_EIO;
        bytes -= n;
    }
    return ZERO3_OK;
}

}  // namespace

extern "C" {

zero3_status zero3_save_shard(const zero3_plan* p, int32_t rank, int64_t t, const float* master,
                              const float* m, const float* v, const char* path,
                              zero3_stream stream) {
    if (!p || !path || rank < 0 || rank >= p->n_ranks || t < 0) return ZERO3_EINVAL;
    if (p->S > 0 && (!master || !m || !v)) return ZERO3_EINVAL;
    const void* arrays[3] = {master, m, v};
    return save_arrays(p, path, kShard, rank, p->S, t, arrays, 3, 4, stream);
}

zero3_status zero3_load_shard(const zero3_plan* p, int32_t rank, int64_t* t, float* master,
                              float* m, float* v, const char* path, zero3_stream stream) {
    if (!p || !path || !t || rank < 0 || rank >= p->n_ranks) return ZERO3_EINVAL;
    if (p->S > 0 && (!master || !m || !v)) return ZERO3_EINVAL;
    void* arrays[3] = {master, m, v};
    return load_arrays(p, path, kShard, rank, p->S, t, arrays, 3, 4, stream);
}

zero3_status zero3_save_persistent(const zero3_plan* p, int64_t t,
                                   const zero3_persist_state* ps, const char* path,
                                   zero3_stream stream) {
    if (!p || !path || !ps || t < 0) return ZERO3_EINVAL;
    if (p->psi_s > 0 && (!ps->master || !ps->m || !ps->v)) return ZERO3_EINVAL;
    const void* arrays[3] = {ps->master, ps->m, ps->v};
    return save_arrays(p, path, kPersist, -1, p->psi_s, t, arrays, 3, 4, stream);
}

zero3_status zero3_load_persistent(const zero3_plan* p, int64_t* t,
                                   const zero3_persist_state* ps, const char* path,
                                   zero3_stream stream) {
    if (!p || !path || !ps || !t) return ZERO3_EINVAL;
    if (p->psi_s > 0 && (!ps->master || !ps->m || !ps->v)) return ZERO3_EINVAL;
    void* arrays[3] = {ps->master, ps->m, ps->v};
    return load_arrays(p, path, kPersist, -1, p->psi_s, t, arrays, 3, 4, stream);
}

zero3_status zero3_save_16bit_weights(const zero3_plan* p, const uint16_t* full,
                                      const uint16_t* persist_param, const char* path,
                                      zero3_stream stream) {
    if (!p || !path) return ZERO3_EINVAL;
    if (p->psi_p > 0 && (!full || !aligned16(full))) return ZERO3_EINVAL;
    if (p->psi_s > 0 && !persist_param) return ZERO3_EINVAL;
    AtomicFile file;
    zero3_status st0 = file.open(path);
    if (st0 != ZERO3_OK) return st0;
    const int64_t total = p->psi_p + p->psi_s;
    const Header h = make_header(p, kWeights16, -1, total, 0);
    if (std::fwrite(&h, sizeof(h), 1, file.f) != 1) return ZERO3_EIO;
    std::vector<char> buf;
    try {
        buf.resize(kStage);
    } catch (const std::bad_alloc&) {
        return ZERO3_ENOMEM;
    }
    // Tensors in list order; a partitioned tensor is contiguous in the flat
    // all-gathered buffer, a persistent one in the persistent copy.
    for (size_t t = 0; t < p->numel.size(); ++t) {
        const uint16_t* src = (p->persistent[t] ? persist_param : full) + p->offset[t];
        zero3_status st = write_device(file.f, src, p->numel[t] * 2, buf, stream);
        if (st != ZERO3_OK) return st;
    }
    return file.commit();
}

zero3_status zero3_merge_shards(const zero3_plan* p, const char* const* shard_paths,
                               const char* persistent_path, const char* out_path) {
    if (!p || !shard_paths || !out_path) return ZERO3_EINVAL;
    if (p->psi_s > 0 && !persistent_path) return ZERO3_EINVAL;
    for (int r = 0; r < p->n_ranks; ++r)
        if (!shard_paths[r]) return ZERO3_EINVAL;
    // open and validate every input before writing anything
    std::vector<File> shards(p->n_ranks);
    int64_t t = -1;
    for (int r = 0; r < p->n_ranks; ++r) {
        Header h;
        zero3_status st =
            open_checked(p, shard_paths[r], kShard, r, p->S, 3 * p->S * 4, shards[r], h);
        if (st != ZERO3_OK) return st;
        if (t >= 0 && h.t != t) return ZERO3_EIO;  // shards of different steps
        t = h.t;
    }
    File pers;
    if (p->psi_s > 0) {
        Header h;
        zero3_status st =
            open_checked(p, persistent_path, kPersist, -1, p->psi_s, 3 * p->psi_s * 4, pers, h);
        if (st != ZERO3_OK) return st;
        if (t >= 0 && h.t != t) return ZERO3_EIO;
        t = h.t;
    }
    AtomicFile out;
    zero3_status st0 = out.open(out_path);
    if (st0 != ZERO3_OK) return st0;
    const Header h = make_header(p, kWeights32, -1, p->psi_p + p->psi_s, t < 0 ? 0 : t);
    if (std::fwrite(&h, sizeof(h), 1, out.f) != 1) return ZERO3_EIO;
    std::vector<char> buf;
    try {
        buf.resize(kStage);
    } catch (const std::bad_alloc&) {
        return ZERO3_ENOMEM;
    }
    // each tensor in list order; a shard file holds master, m, v: the master
    // array starts right after the header
    for (size_t ti = 0; ti < p->numel.size(); ++ti) {
        zero3_status st = ZERO3_OK;
        if (p->persistent[ti]) {
            st = copy_range(pers.f, static_cast<int64_t>(sizeof(Header)) + p->offset[ti] * 4,
                            p->numel[ti] * 4, out.f, buf);
        } else {
            for (int64_t sgi = p->seg_begin[ti]; sgi < p->seg_begin[ti + 1] && st == ZERO3_OK; ++sgi) {
                const zero3_segment& sg = p->segs[sgi];
                st = copy_range(shards[sg.rank].f,
                                static_cast<int64_t>(sizeof(Header)) + sg.shard_off * 4,
                                sg.len * 4, out.f, buf);
            }
        }
        if (st != ZERO3_OK) return st;
    }
    return out.commit();
}

}  // extern "C"
