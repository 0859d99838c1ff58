// wa_prep.cu — q/k preparation and KV append (the step that fills the caches).
//
// Two preparations, per head of d values:
//   RMSNorm (page "Exact Numerical Contract", section "Preparation"):
//     y = x * (1 / sqrt(sum(x^2) / d + 1e-5)) in fp32, rounded once to bf16.
//   L2 + RoPE (TensorFold pull request #1257, section "What the kernel computes"):
//     r = bf16(rotate_half(x, fl32(pos * inv_freq)))   fp32 cosf/sinf
//     n = bf16(r * (1 / sqrt(sum(r^2) + 1e-6)))
//     q = bf16(q_scale * n) for query heads, k = n for key heads.
// v is copied as is; k and v land in ring slot pos mod ring.
//
// HBM-bound elementwise work with one reduction per head.  One warp per
// (token, head); lane l holds dims [E l, E l + E) and [d/2 + E l, d/2 + E l + E)
// (E = d / 64), so each rotate-half pair sits in one lane and both halves load
// as coalesced segments.  The sum of squares is a fixed xor butterfly, so every
// lane holds the same bits and the result does not depend on the launch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "wa.h"
#include "wa_internal.h"

namespace wa {

namespace {

constexpr int kPrepWarps = 8;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// Rounds an fp32 value to bf16 and back (a rounding point of the preparation).
__device__ __forceinline__ float round_bf16(float x) { return bf16_bits_to_f32(f32_to_bf16_bits(x)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

// E consecutive bf16 values (E = 2 or 4) as 32- or 64-bit loads and stores.
template <int E>
__device__ __forceinline__ void load_e(const uint16_t* p, float (&x)[E]) {
    if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        x[0] = bf16_bits_to_f32(u.x & 0xFFFFu); x[1] = bf16_bits_to_f32(u.x >> 16);
        x[2] = bf16_bits_to_f32(u.y & 0xFFFFu); x[3] = bf16_bits_to_f32(u.y >> 16);
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        x[0] = bf16_bits_to_f32(u & 0xFFFFu); x[1] = bf16_bits_to_f32(u >> 16);
    }
}

template <int E>
__device__ __forceinline__ void store_e(uint16_t* p, const float (&y)[E]) {
    if constexpr (E == 4) {
        uint2 u;
        u.x = f32_to_bf16_bits(y[0]) | (f32_to_bf16_bits(y[1]) << 16);
        u.y = f32_to_bf16_bits(y[2]) | (f32_to_bf16_bits(y[3]) << 16);
        *reinterpret_cast<uint2*>(p) = u;
    } else {
        *reinterpret_cast<uint32_t*>(p) = f32_to_bf16_bits(y[0]) | (f32_to_bf16_bits(y[1]) << 16);
    }
}

template <int E>
__device__ __forceinline__ void copy_e(uint16_t* dst, const uint16_t* src) {
    if constexpr (E == 4) *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(src);
    else *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
}

struct PrepParams {
    const uint16_t* src;
    const int32_t* pos;
    const float* q_scale;
    const float* inv_freq;
    uint16_t* q_out;
    uint16_t* k_ring;
    uint16_t* v_ring;
    int* status;
    int64_t src_tok, q_tok, ring_row, slot;
    int n, hq, hkv, ring, mode;
};

template <int D>
__global__ void __launch_bounds__(kPrepWarps * 32) prep_kernel(const PrepParams p) {
    constexpr int E = D / 64;
    constexpr int H = D / 2;
    const int heads = p.hq + 2 * p.hkv;
    const int64_t job = static_cast<int64_t>(blockIdx.x) * kPrepWarps + (threadIdx.x >> 5);
    if (job >= static_cast<int64_t>(p.n) * heads) return;   // warp-uniform
    const int lane = threadIdx.x & 31;
    const int t = static_cast<int>(job / heads), hh = static_cast<int>(job % heads);
    const int pos = p.pos[t];
    if (pos < 0) {
        if (hh == 0 && lane == 0) atomicOr(p.status, WA_STATUS_BAD_POS);
        return;
    }
    const uint16_t* x_head = p.src + t * p.src_tok + static_cast<int64_t>(hh) * D;
    const int64_t slot_off = t * p.ring_row + static_cast<int64_t>(pos % p.ring) * p.slot;
    const int j0 = lane * E;   // this lane's dims: [j0, j0 + E) and [H + j0, H + j0 + E)

    if (hh >= p.hq + p.hkv) {   // value head: copied as is
        if (p.v_ring) {
            uint16_t* dst = p.v_ring + slot_off + static_cast<int64_t>(hh - p.hq - p.hkv) * D;
            copy_e<E>(dst + j0, x_head + j0);
            copy_e<E>(dst + H + j0, x_head + H + j0);
        }
        return;
    }
    const bool is_q = hh < p.hq;
    float lo[E], hi[E];
    load_e<E>(x_head + j0, lo);
    load_e<E>(x_head + H + j0, hi);

    if (p.mode == WA_PREP_RMSNORM) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = __fmaf_rn(lo[e], lo[e], __fmaf_rn(hi[e], hi[e], ss));
        ss = warp_sum(ss);
        // 1/d is a power of two, so the mean is exact; one IEEE square root and one IEEE divide
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fmaf_rn(ss, 1.0f / D, 1e-5f)));
#pragma unroll
        for (int e = 0; e < E; ++e) {
            lo[e] = __fmul_rn(lo[e], inv);
            hi[e] = __fmul_rn(hi[e], inv);
        }
    } else {
        const float fp = static_cast<float>(pos);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float ang = __fmul_rn(fp, p.inv_freq[j0 + e]);   // fl32(pos * inv)
            float s, c;
            sincosf(ang, &s, &c);
            const float a = lo[e], b = hi[e];
            lo[e] = round_bf16(__fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s)));
            hi[e] = round_bf16(__fadd_rn(__fmul_rn(b, c), __fmul_rn(a, s)));
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = __fmaf_rn(lo[e], lo[e], __fmaf_rn(hi[e], hi[e], ss));
        ss = warp_sum(ss);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ss, 1e-6f)));
#pragma unroll
        for (int e = 0; e < E; ++e) {
            lo[e] = __fmul_rn(lo[e], inv);
            hi[e] = __fmul_rn(hi[e], inv);
        }
        if (is_q && p.q_scale) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                lo[e] = __fmul_rn(round_bf16(lo[e]), p.q_scale[j0 + e]);
                hi[e] = __fmul_rn(round_bf16(hi[e]), p.q_scale[H + j0 + e]);
            }
        }
    }
    uint16_t* dst = is_q ? p.q_out + t * p.q_tok + static_cast<int64_t>(hh) * D
                         : p.k_ring + slot_off + static_cast<int64_t>(hh - p.hq) * D;
    store_e<E>(dst + j0, lo);
    store_e<E>(dst + H + j0, hi);
}

}  // namespace

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
    PrepParams p{};
    p.src = static_cast<const uint16_t*>(a.src);
    p.pos = a.pos;
    p.q_scale = a.q_scale;
    p.inv_freq = a.inv_freq;
    p.q_out = static_cast<uint16_t*>(a.q_out);
    p.k_ring = static_cast<uint16_t*>(a.k_ring);
    p.v_ring = static_cast<uint16_t*>(a.v_ring);
    p.status = &a.hdr->status;
    p.src_tok = a.src_tok; p.q_tok = a.q_tok; p.ring_row = a.ring_row; p.slot = a.slot;
    p.n = a.n; p.hq = a.hq; p.hkv = a.hkv; p.ring = a.ring; p.mode = a.mode;
    const int64_t jobs = static_cast<int64_t>(a.n) * (a.hq + 2 * a.hkv);
    const int64_t blocks = (jobs + kPrepWarps - 1) / kPrepWarps;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    if (a.d == 256) prep_kernel<256><<<static_cast<unsigned>(blocks), kPrepWarps * 32, 0, s>>>(p);
    else prep_kernel<128><<<static_cast<unsigned>(blocks), kPrepWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace wa
