// Device helpers shared by the streaming kernels (kernels.cu) and the piece
// kernel (pieces.cu): block size, programmatic dependent launch, bf16
// conversion and packing, streaming 16-byte accesses, the launch helper.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace z3 {
namespace {

constexpr int kThreads = 256;

// Programmatic dependent launch.  Every kernel of this library is launched with
// programmatic stream serialization, so it may be scheduled while the
// previous kernel of the stream drains.  Each thread therefore waits for the
// previous grids to complete (and their writes to become visible) before its
// first memory access, which keeps plain stream order for the data; what
// overlaps is the launch and block dispatch of this grid with the previous
// grid's tail.  Without a programmatic predecessor the wait returns at once.
__device__ __forceinline__ void wait_prior_grids() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next programmatic launch of the stream be scheduled.
__device__ __forceinline__ void allow_next_grid() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Two binary32 values -> packed bf16 pair, round to nearest even (hardware
// conversion); `lo` lands in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint16_t to_bf16(float x) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
    return r;
}

// Streaming (evict-first) 16-byte accesses: every byte is touched once.
__device__ __forceinline__ uint4 ldcs16(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void stcs16(void* p, uint4 x) { __stcs(reinterpret_cast<uint4*>(p), x); }

__device__ __forceinline__ void unpack8(const uint4& r, float* f) {
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x);
    f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z);
    f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

// Launch with programmatic stream serialization (see wait_prior_grids).
template <typename Args>
cudaError_t launch_programmatic(void (*kernel)(Args), int grid, const Args& a,
                                cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace
}  // namespace z3
