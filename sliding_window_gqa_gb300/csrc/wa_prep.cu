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
// HBM-bound elementwise work with one reduction per head.  A head is served by
// L = d/16 lanes, each holding 8 dims of the low half and the same 8 dims of the
// high half (so every rotate-half pair sits in one lane, and each lane moves
// 16-byte pieces).  A warp takes P = 32/L heads per pass and kPasses passes of
// one token, with every pass's loads issued before any arithmetic, so that
// enough bytes are in flight to cover DRAM latency.  The angles' sines and
// cosines depend only on the token and the lane's dims: computed once per warp.
// The sum of squares is a fixed xor butterfly within the L lanes, so the result
// does not depend on the launch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "wa.h"
#include "wa_internal.h"

namespace wa {

namespace {

constexpr int kPrepWarps = 8;
constexpr int kPasses = 4;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// Rounds an fp32 value to bf16 and back (a rounding point of the preparation).
__device__ __forceinline__ float round_bf16(float x) { return __uint_as_float(f32_to_bf16_bits(x) << 16); }

__device__ __forceinline__ void unpack8(const uint4& u, float (&x)[8]) {
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint4 pack8(const float (&y)[8]) {
    uint4 u;
    u.x = f32_to_bf16_bits(y[0]) | (f32_to_bf16_bits(y[1]) << 16);
    u.y = f32_to_bf16_bits(y[2]) | (f32_to_bf16_bits(y[3]) << 16);
    u.z = f32_to_bf16_bits(y[4]) | (f32_to_bf16_bits(y[5]) << 16);
    u.w = f32_to_bf16_bits(y[6]) | (f32_to_bf16_bits(y[7]) << 16);
    return u;
}

// Sum over the L lanes serving one head (an xor butterfly, the same bits in every lane).
template <int L>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
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
    int n, hq, hkv, ring, mode, warps_per_token;
};

template <int D>
__global__ void __launch_bounds__(kPrepWarps * 32) prep_kernel(const PrepParams p) {
    constexpr int H = D / 2;
    constexpr int L = D / 16;          // lanes per head
    constexpr int P = 32 / L;          // heads per pass
    constexpr int HPW = P * kPasses;   // query/key heads per warp
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * kPrepWarps + (threadIdx.x >> 5);
    if (wid >= static_cast<int64_t>(p.n) * p.warps_per_token) return;   // warp-uniform
    const int lane = threadIdx.x & 31;
    const int t = static_cast<int>(wid / p.warps_per_token);
    const int sub = static_cast<int>(wid % p.warps_per_token);
    const int pos = p.pos[t];
    if (pos < 0) {
        if (sub == 0 && lane == 0) atomicOr(p.status, WA_STATUS_BAD_POS);
        return;
    }
    const int nqk = p.hq + p.hkv;
    const int li = lane % L, hp = lane / L;
    const int j0 = 8 * li;             // this lane's dims: [j0, j0 + 8) and [H + j0, H + j0 + 8)
    const uint16_t* row = p.src + t * p.src_tok;
    const int64_t slot_off = t * p.ring_row + static_cast<int64_t>(pos % p.ring) * p.slot;

    if (sub * HPW < nqk) {
        // ---- query and key heads: all loads first
        uint4 raw[kPasses][2];
#pragma unroll
        for (int u = 0; u < kPasses; ++u) {
            const int hh = sub * HPW + u * P + hp;
            if (hh < nqk) {
                raw[u][0] = *reinterpret_cast<const uint4*>(row + static_cast<int64_t>(hh) * D + j0);
                raw[u][1] = *reinterpret_cast<const uint4*>(row + static_cast<int64_t>(hh) * D + H + j0);
            } else {
                raw[u][0] = raw[u][1] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        float c[8], s[8];
        if (p.mode == WA_PREP_L2_ROPE) {
            const float fp = static_cast<float>(pos);
#pragma unroll
            for (int e = 0; e < 8; ++e) sincosf(__fmul_rn(fp, p.inv_freq[j0 + e]), &s[e], &c[e]);   // fl32(pos * inv)
        }
#pragma unroll
        for (int u = 0; u < kPasses; ++u) {
            const int hh = sub * HPW + u * P + hp;
            float lo[8], hi[8];
            unpack8(raw[u][0], lo);
            unpack8(raw[u][1], hi);
            float inv;
            if (p.mode == WA_PREP_RMSNORM) {
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = __fmaf_rn(lo[e], lo[e], __fmaf_rn(hi[e], hi[e], ss));
                ss = group_sum<L>(ss);
                // 1/d is a power of two, so the mean is exact; one IEEE square root and one IEEE divide
                inv = __fdiv_rn(1.0f, __fsqrt_rn(__fmaf_rn(ss, 1.0f / D, 1e-5f)));
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float a = lo[e], b = hi[e];
                    lo[e] = round_bf16(__fsub_rn(__fmul_rn(a, c[e]), __fmul_rn(b, s[e])));
                    hi[e] = round_bf16(__fadd_rn(__fmul_rn(b, c[e]), __fmul_rn(a, s[e])));
                }
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = __fmaf_rn(lo[e], lo[e], __fmaf_rn(hi[e], hi[e], ss));
                ss = group_sum<L>(ss);
                inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ss, 1e-6f)));
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                lo[e] = __fmul_rn(lo[e], inv);
                hi[e] = __fmul_rn(hi[e], inv);
            }
            if (hh >= nqk) continue;
            const bool is_q = hh < p.hq;
            if (is_q && p.mode == WA_PREP_L2_ROPE && p.q_scale) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    lo[e] = __fmul_rn(round_bf16(lo[e]), p.q_scale[j0 + e]);
                    hi[e] = __fmul_rn(round_bf16(hi[e]), p.q_scale[H + j0 + e]);
                }
            }
            uint16_t* dst = is_q ? p.q_out + t * p.q_tok + static_cast<int64_t>(hh) * D
                                 : p.k_ring + slot_off + static_cast<int64_t>(hh - p.hq) * D;
            *reinterpret_cast<uint4*>(dst + j0) = pack8(lo);
            *reinterpret_cast<uint4*>(dst + H + j0) = pack8(hi);
        }
    } else if (p.v_ring) {
        // ---- value heads: copied as is, 16 bytes a lane
        const int vw = sub - (nqk + HPW - 1) / HPW;   // this warp's share of the token's value heads
        const int nv = p.hkv * D / 8;                 // 16-byte pieces
        const int vwarps = p.warps_per_token - (nqk + HPW - 1) / HPW;
        const uint16_t* vsrc = row + static_cast<int64_t>(nqk) * D;
        uint16_t* vdst = p.v_ring + slot_off;
        for (int i = vw * 32 + lane; i < nv; i += vwarps * 32)
            *reinterpret_cast<uint4*>(vdst + 8 * i) = *reinterpret_cast<const uint4*>(vsrc + 8 * i);
    }
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
    const int hpw = (32 / (a.d / 16)) * kPasses;
    const int qk_warps = (a.hq + a.hkv + hpw - 1) / hpw;
    // value heads: up to one warp per 512 bytes of the token's values
    const int v_warps = a.v_ring ? (a.hkv * a.d * 2 + 511) / 512 : 0;
    p.warps_per_token = qk_warps + v_warps;
    const int64_t warps = static_cast<int64_t>(a.n) * p.warps_per_token;
    const int64_t blocks = (warps + kPrepWarps - 1) / kPrepWarps;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    if (a.d == 256) prep_kernel<256><<<static_cast<unsigned>(blocks), kPrepWarps * 32, 0, s>>>(p);
    else prep_kernel<128><<<static_cast<unsigned>(blocks), kPrepWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace wa
