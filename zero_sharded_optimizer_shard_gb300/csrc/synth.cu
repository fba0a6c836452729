// Device side of the seeded counter-based input generator, built as its own
// library (libzero3_synth.so).  It draws numbers only and holds none of the
// optimizer's arithmetic.  Definition (shared with the host generator, which
// is written independently in Python):
//
//   mix64 = SplitMix64 output function (Steele, Lea, Flood, OOPSLA 2014)
//   key   = mix64(mix64(mix64(seed + G*(stream+1)) + G*(step+1)) + G*(rank+1))
//   draw(index, j) = mix64(key + G*(8*index + j + 1)),  G = 0x9e3779b97f4a7c15
//   normal: Irwin-Hall(12) from the 24-bit fields (bits 40..63 and 8..31) of
//   draws 0..5, x = (f32(sum) * 2^-24 - 6) * f32(sigma_eff), binary32 RNE ops;
//   sigma_eff = outlier_sigma when (draw 6 >> 32) < floor(outlier_p * 2^32);
//   bf16 sample = upper 16 bits of x.
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr uint64_t kGolden = 0x9e3779b97f4a7c15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

uint64_t make_key(uint64_t seed, int64_t stream, int64_t step, int64_t rank) {
    const uint64_t k0 = mix64(seed + kGolden * static_cast<uint64_t>(stream + 1));
    const uint64_t k1 = mix64(k0 + kGolden * static_cast<uint64_t>(step + 1));
    return mix64(k1 + kGolden * static_cast<uint64_t>(rank + 1));
}

__global__ void normal_kernel(uint64_t key, int64_t index0, int64_t n, float sigma,
                              uint64_t outlier_thr, float outlier_sigma, int bf16, void* out) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n;
         k += stride) {
        const uint64_t base = key + kGolden * (8ull * static_cast<uint64_t>(index0 + k));
        uint64_t s = 0;
#pragma unroll
        for (int j = 0; j < 6; ++j) {
            const uint64_t d = mix64(base + kGolden * static_cast<uint64_t>(j + 1));
            s += (d >> 40) & 0xffffffull;
            s += (d >> 8) & 0xffffffull;
        }
        float sig = sigma;
        if (outlier_thr) {
            const uint64_t d6 = mix64(base + kGolden * 7ull);
            if ((d6 >> 32) < outlier_thr) sig = outlier_sigma;
        }
        float x = __ll2float_rn(static_cast<long long>(s));
        x = __fmul_rn(x, 5.9604644775390625e-08f);  // 2^-24, exact
        x = __fsub_rn(x, 6.0f);
        x = __fmul_rn(x, sig);
        if (bf16)
            static_cast<uint16_t*>(out)[k] = static_cast<uint16_t>(__float_as_uint(x) >> 16);
        else
            static_cast<float*>(out)[k] = x;
    }
}

}  // namespace

extern "C" {

// Fills out[k] (k < n) with the sample at flat index index0 + k.
// out_bf16 != 0: uint16 bf16 patterns, else binary32.  Returns a cudaError_t.
int zero3synth_normal(uint64_t seed, int64_t stream_id, int64_t step, int64_t rank, int64_t index0,
                      int64_t n, double sigma, double outlier_p, double outlier_sigma,
                      int32_t out_bf16, void* out, cudaStream_t stream) {
    if (n <= 0) return 0;
    if (!out || index0 < 0) return static_cast<int>(cudaErrorInvalidValue);
    const uint64_t key = make_key(seed, stream_id, step, rank);
    const uint64_t thr = outlier_p > 0.0 ? static_cast<uint64_t>(outlier_p * 4294967296.0) : 0;
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t need = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    const int grid = static_cast<int>(need < cap ? need : cap);
    normal_kernel<<<grid, 256, 0, stream>>>(key, index0, n, static_cast<float>(sigma), thr,
                                            static_cast<float>(outlier_sigma), out_bf16, out);
    return static_cast<int>(cudaGetLastError());
}

}  // extern "C"
