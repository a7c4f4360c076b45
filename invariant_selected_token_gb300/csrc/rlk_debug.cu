// Diagnostic sweeps of the contract's primitives.
//
// The numeric contract fixes its own exp, log and rsqrt (written with
// explicit round-to-nearest operations), and the CPU emulator restates them
// in C.  rlk_debug_primitive_hash evaluates one primitive on the GPU over a
// contiguous range of fp32 bit patterns and folds the results into one
// position-weighted 64-bit sum, sum_i (bits(f(x_i)) + 0x9E3779B9) (2 i + 1)
// mod 2^64, which the emulator forms the same way: a single differing output
// changes the sum (its weight is odd), so equal sums over a whole input
// range show the two implementations agree bit for bit there.  Primitive 1
// is exp evaluated two lanes at a time (the packed form the kernels use).
#include <cstdint>
#include <cuda_runtime.h>

#include "rlk_contract.cuh"
#include "rlk_internal.h"

namespace rlk {
namespace {

__device__ __forceinline__ uint64_t term(float y, uint64_t i) {
    return (static_cast<uint64_t>(__float_as_uint(y)) + 0x9E3779B9ull) * (2ull * i + 1ull);
}

template <int kWhich>
__global__ void __launch_bounds__(256)
    k_primitive_hash(uint32_t first, uint64_t count, unsigned long long* out) {
    uint64_t h = 0;
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    const uint64_t start = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (kWhich == 1) {
        const uint64_t pairs = (count + 1) / 2;
        for (uint64_t p = start; p < pairs; p += stride) {
            const uint64_t i0 = 2 * p;
            const bool two = i0 + 1 < count;
            const float x0 = __uint_as_float(first + static_cast<uint32_t>(i0));
            const float x1 = two ? __uint_as_float(first + static_cast<uint32_t>(i0 + 1)) : 0.0f;
            float y0, y1;
            f2_unpack(contract_exp_x2(f2_pack(x0, x1)), y0, y1);
            h += term(y0, i0);
            if (two) h += term(y1, i0 + 1);
        }
    } else {
        for (uint64_t i = start; i < count; i += stride) {
            const float x = __uint_as_float(first + static_cast<uint32_t>(i));
            const float y = kWhich == 0 ? contract_exp(x) : kWhich == 2 ? contract_log(x)
                                                                        : contract_rsqrt(x);
            h += term(y, i);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(out, static_cast<unsigned long long>(h));
}

template <int kWhich>
cudaError_t launch_hash(uint32_t first, uint64_t count, unsigned long long* out, int blocks,
                        cudaStream_t stream) {
    k_primitive_hash<kWhich><<<blocks, 256, 0, stream>>>(first, count, out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_primitive_hash(int which, uint32_t first, uint64_t count, uint64_t* out,
                                  int num_sms, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(uint64_t), stream);
    if (e != cudaSuccess || count == 0) return e;
    unsigned long long* o = reinterpret_cast<unsigned long long*>(out);
    const int blocks = num_sms * 8;
    switch (which) {
        case 0: return launch_hash<0>(first, count, o, blocks, stream);
        case 1: return launch_hash<1>(first, count, o, blocks, stream);
        case 2: return launch_hash<2>(first, count, o, blocks, stream);
        case 3: return launch_hash<3>(first, count, o, blocks, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rlk
