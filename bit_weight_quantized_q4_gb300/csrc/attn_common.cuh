// attn_common.cuh -- register-level pieces of decode attention shared by the
// standalone attention kernel (attn_kernel.cu) and the persistent decode
// step's attention job (step_attn.cuh): RoPE of a head held across a warp,
// row loads, and the transpose-reduce of 32 partial dot products.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace q4 {
namespace dev {

// RoPE of a head vector held DL = D/32 elements per lane (lane l holds
// elements l*DL .. l*DL+DL-1): element e pairs with e + D/2, which lane l ^ 16
// holds; (a, b) -> (a c - b s, b c + a s) with the table row of the position.
template <int DL>
__device__ __forceinline__ void rope_lane(float (&x)[DL], const float *cosr, const float *sinr, int lane) {
    constexpr int HALF = 16 * DL;
#pragma unroll
    for (int j = 0; j < DL; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, x[j], 16);
        const int jj = (lane * DL + j) % HALF;
        const float c = __ldg(cosr + jj), s = __ldg(sinr + jj);
        x[j] = lane < 16 ? x[j] * c - other * s : x[j] * c + other * s;
    }
}

template <int DL>
__device__ __forceinline__ void load_row(float (&x)[DL], const float *src) {
    if constexpr (DL == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(src);
        x[0] = v.x;
        x[1] = v.y;
    } else {
        const float4 v = *reinterpret_cast<const float4 *>(src);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
    }
}

// N consecutive floats of shared memory (N a power of two), in 16-byte loads
// where they fit.
template <int N>
__device__ __forceinline__ void load_vec(float (&x)[N], const float *src) {
    if constexpr (N >= 4) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(src + i);
            x[i] = v.x;
            x[i + 1] = v.y;
            x[i + 2] = v.z;
            x[i + 3] = v.w;
        }
    } else if constexpr (N == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(src);
        x[0] = v.x;
        x[1] = v.y;
    } else {
        x[0] = src[0];
    }
}

// 32 partial sums per lane -> lane l holds the warp-wide sum of value l
// (recursive halving: each round a lane keeps the half of its values whose
// index bit matches its lane bit and adds its partner's share of it).
__device__ __forceinline__ float transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// Start pulling `bytes` (16-byte aligned, a multiple of 16) of global memory
// into L2 and go on.  A hint only: every later read of those bytes goes
// through L2, the point of coherence, so it sees every write made since.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

}  // namespace dev
}  // namespace q4
