// wa_decode.cu — decode form: per-chunk partials, then an ordered merge.
//
// TensorFold pull request #1123 ("window_attention at head dim 256"),
// section "What this changes", bullet "Decode": 256-key chunks at absolute
// key positions, one block per (row, key head, chunk), fp32 scores and
// probabilities, a chunk max m_c, p = exp(s - m_c), l_c = sum p,
// o_c = sum p v, then a merge o = sum_c a_c o_c / sum_c a_c l_c with
// a_c = exp(m_c - M), as an fma chain over the chunks in order.  Chunks that
// hold none of a row's keys are skipped, so a row's bits do not depend on
// the batch, the row's slot or the ring length.
//
// GB300 design: the CTA holds every query head of its key-head group, so K
// and V are read from HBM once per group.  A producer warp stages 32-key runs
// into a ring of shared-memory stages against mbarriers: a run whose keys are
// all visible and sit in consecutive ring slots is one TMA tensor box (32 key
// rows of one head); a run cut by the window or the ring's end is copied row
// by row with cp.async.bulk.  Eight
// consumer warps each own one 32-key run of the chunk.  Scores use an fp32
// fma chain over a lane's d/32 dims, then a butterfly over the 32 lanes
// (every lane ends with identical bits); o is an fma chain in key order per
// run, and the eight run partials are added in run order.
#include <cuda_bf16.h>

#include "wa_internal.h"
#include "wa_ptx.cuh"

namespace wa {

namespace {

constexpr int kRun = 32;                   // keys per run: one consumer warp each
constexpr int kRuns = kChunk / kRun;       // 8
constexpr int kConsumerWarps = kRuns;
constexpr int kPartThreads = (kConsumerWarps + 1) * 32;

template <int D, int G>  // G: the head-group bucket (a power of two >= the group size)
struct PartCfg {
    static constexpr int DPL = D / 32;                  // dims per lane
    static constexpr int ROWB = D * 2;                  // bytes of one key row
    static constexpr int STAGE_B = kRun * ROWB;         // one run of K or V
    static constexpr int OBUF_B = kRuns * G * D * 4;    // run partials, aliased on the stage ring
    static constexpr int STAGES = (OBUF_B / STAGE_B) > 4 ? (OBUF_B / STAGE_B) : 4;
    static constexpr int RING_B = STAGES * STAGE_B;
    static constexpr int SC_OFF = RING_B;                       // scores, then p: [256][G] fp32
    static constexpr int MW_OFF = SC_OFF + kChunk * G * 4;      // run maxima [8][G]
    static constexpr int LW_OFF = MW_OFF + kRuns * G * 4;       // run sums [8][G]
    static constexpr int BAR_OFF = (LW_OFF + kRuns * G * 4 + 15) & ~15;
    static constexpr int NLOADS = 2 * kRuns;                    // K runs, then V runs
    static constexpr int SMEM = BAR_OFF + 2 * NLOADS * 8;        // full[t], consumed[t]
    static constexpr int MIN_BLOCKS = (G <= 4) ? 2 : 1;
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void bf16x4_to_f32(const uint2 u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xFFFF0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xFFFF0000u);
}

// This lane's d/32 dims of a d-element bf16 row, as fp32.
template <int D>
__device__ __forceinline__ void load_lane_dims(const void* row, int lane, float (&f)[D / 32]) {
    if constexpr (D == 256) {
        const uint4 u = reinterpret_cast<const uint4*>(row)[lane];
        bf16x8_to_f32(u, f);
    } else {
        const uint2 u = reinterpret_cast<const uint2*>(row)[lane];
        bf16x4_to_f32(u, f);
    }
}

__device__ __forceinline__ float warp_sum_butterfly(float x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    return x;
}

// Clamp a device-side position into the valid range; report once per row.
__device__ __forceinline__ int checked_pos(const int32_t* pos, int r, int win, int ring, int* status, bool report) {
    int p = pos[r];
    if (p < 0) {
        if (report) atomicOr(status, WA_STATUS_BAD_POS);
        p = 0;
    }
    if (win == 0 && p >= ring) {
        if (report) atomicOr(status, WA_STATUS_BAD_POS);
        p = ring - 1;
    }
    return p;
}

// K and V rings as 4-D tensors (d, key head, slot, row); one box is one 32-key run of one head.
struct RingMaps {
    CUtensorMap tk, tv;
};

template <int D, int G>
__global__ void __launch_bounds__(kPartThreads, PartCfg<D, G>::MIN_BLOCKS)
decode_part_kernel(const __grid_constant__ RingMaps maps,
                   const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                   const __nv_bfloat16* __restrict__ v, const int32_t* __restrict__ pos,
                   int hq, int hkv, int gsize, int win, int ring, float scale, int cmax,
                   float* __restrict__ part, int* __restrict__ status) {
    using C = PartCfg<D, G>;
    constexpr int DPL = C::DPL;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int ci = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
    const int p = checked_pos(pos, r, win, ring, status, ci == 0 && g == 0 && threadIdx.x == 0);
    const int lo = win > 0 ? max(0, p - win + 1) : 0;
    const int c = lo / kChunk + ci;
    if (c > p / kChunk) return;                       // no key of this row in the chunk
    const int cbase = c * kChunk;
    const int kb = max(lo, cbase), ke = min(p, cbase + kChunk - 1);
    const int w0 = (kb - cbase) / kRun, w1 = (ke - cbase) / kRun, nr = w1 - w0 + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint8_t* stage = smem;
    float* sc = reinterpret_cast<float*>(smem + C::SC_OFF);
    float* mw = reinterpret_cast<float*>(smem + C::MW_OFF);
    float* lw = reinterpret_cast<float*>(smem + C::LW_OFF);
    // Load t (K run w0+t for t < nr, then V run w0+t-nr) lands in stage t % STAGES.
    // Each load has its own single-use barriers: full[t] (bytes landed) and
    // consumed[t] (stage free again), so every wait is on phase 0 of a fresh
    // barrier and no waiter can confuse one use of a stage with another.
    const uint32_t bar_full = smem_u32(smem + C::BAR_OFF);
    const uint32_t bar_used = bar_full + 8 * C::NLOADS;

    if (threadIdx.x == 0) {
        for (int t = 0; t < C::NLOADS; ++t) {
            mbar_init(bar_full + 8 * t, 1);
            mbar_init(bar_used + 8 * t, 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    const size_t row0 = static_cast<size_t>(r) * ring;   // first key row of this row's ring

    if (warp == kConsumerWarps) {
        // ---------------- producer: K runs w0..w1, then V runs w0..w1 ----------------
        const uint64_t pol = policy_evict_first();
        int issued = 0;
        bool ok = true;
        for (int t = 0; t < 2 * nr; ++t) {
            const int st = t % C::STAGES;
            if (t >= C::STAGES && !warp_wait(bar_used + 8 * (t - C::STAGES), 0, status)) { ok = false; break; }
            const int run = w0 + (t % nr);
            const __nv_bfloat16* src_base = (t < nr) ? k : v;
            const int rb = cbase + run * kRun;
            const int a = max(kb, rb), b = min(ke, rb + kRun - 1);
            const int j = rb + lane;
            const int slot_rb = rb % ring;
            if (a == rb && b == rb + kRun - 1 && slot_rb + kRun <= ring) {
                // a whole run in consecutive slots: one tensor box of 32 key rows
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar_full + 8 * t, static_cast<uint32_t>(kRun * C::ROWB));
                    tma_load_4d(smem_u32(stage + st * C::STAGE_B), (t < nr) ? &maps.tk : &maps.tv, 0, g, slot_rb, r,
                                bar_full + 8 * t, pol);
                }
            } else {
                // a run cut by the window or by the end of the ring: one bulk copy per visible key row
                if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * t, static_cast<uint32_t>((b - a + 1) * C::ROWB));
                __syncwarp();
                if (j >= a && j <= b) {
                    const __nv_bfloat16* src = src_base + ((row0 + static_cast<size_t>(j % ring)) * hkv + g) * D;
                    bulk_g2s(smem_u32(stage + st * C::STAGE_B + lane * C::ROWB), src, C::ROWB, bar_full + 8 * t, pol);
                }
            }
            issued = t + 1;
        }
        // Let the copies already issued land before this warp exits, whichever role stopped early
        // (when every load was consumed these barriers have completed and the waits return at once).
        if (lane == 0)
            for (int t = max(0, issued - C::STAGES); t < issued; ++t) mbar_wait(bar_full + 8 * t, 0, status);
        (void)ok;
        return;
    }

    // ---------------- consumers: warp w owns run w of the chunk ----------------
    const int w = warp;
    const bool active = (w >= w0) && (w <= w1);
    const int rb = cbase + w * kRun;
    const int a = max(kb, rb), b = min(ke, rb + kRun - 1);
    bool ok = true;

    float qf[G][DPL];
    {
        const __nv_bfloat16* qrow = q + (static_cast<size_t>(r) * hq + static_cast<size_t>(g) * gsize) * D;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            if (h < gsize) {
                load_lane_dims<D>(qrow + h * D, lane, qf[h]);
            } else {
#pragma unroll
                for (int e = 0; e < DPL; ++e) qf[h][e] = 0.f;   // bucket slot without a head
            }
        }
    }

    float mrun[G];
#pragma unroll
    for (int h = 0; h < G; ++h) mrun[h] = -INFINITY;

    if (active) {
        const int t = w - w0;
        const int st = t % C::STAGES;
        ok = warp_wait(bar_full + 8 * t, 0, status);
        if (ok) {
            const uint8_t* base = stage + st * C::STAGE_B;
            for (int jj = a - rb; jj <= b - rb; ++jj) {
                float kf[DPL];
                load_lane_dims<D>(base + jj * C::ROWB, lane, kf);
                float s[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float acc = qf[h][0] * kf[0];
#pragma unroll
                    for (int e = 1; e < DPL; ++e) acc = fmaf(qf[h][e], kf[e], acc);
                    s[h] = warp_sum_butterfly(acc) * scale;
                    mrun[h] = fmaxf(mrun[h], s[h]);
                }
                if (lane == 0) {
#pragma unroll
                    for (int h = 0; h < G; ++h) sc[(w * kRun + jj) * G + h] = s[h];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_used + 8 * t);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) mw[w * G + h] = mrun[h];
    }
    named_bar_sync(1, kConsumerWarps * 32);

    float m[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float x = mw[h];
        for (int ww = 1; ww < kRuns; ++ww) x = fmaxf(x, mw[ww * G + h]);
        m[h] = x;
    }

    float acc[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
    float lrun[G];
#pragma unroll
    for (int h = 0; h < G; ++h) lrun[h] = 0.f;

    if (active && ok) {
        const int j = rb + lane;
        const bool vis = (j >= a) && (j <= b);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float pr = vis ? expf(sc[(w * kRun + lane) * G + h] - m[h]) : 0.f;
            lrun[h] = warp_sum_butterfly(pr);
            if (vis) sc[(w * kRun + lane) * G + h] = pr;
        }
        __syncwarp();
        const int t = nr + (w - w0);
        const int st = t % C::STAGES;
        ok = warp_wait(bar_full + 8 * t, 0, status);
        if (ok) {
            const uint8_t* base = stage + st * C::STAGE_B;
            for (int jj = a - rb; jj <= b - rb; ++jj) {
                float vf[DPL];
                load_lane_dims<D>(base + jj * C::ROWB, lane, vf);
                const float* pj = sc + (w * kRun + jj) * G;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float ph = pj[h];
#pragma unroll
                    for (int e = 0; e < DPL; ++e) acc[h][e] = fmaf(ph, vf[e], acc[h][e]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_used + 8 * t);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) lw[w * G + h] = lrun[h];
    }
    named_bar_sync(1, kConsumerWarps * 32);   // every V run consumed: the stage ring is free

    float* obuf = reinterpret_cast<float*>(stage);   // [8][G][D]
    if (ok) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < DPL; ++e) obuf[(w * G + h) * D + lane * DPL + e] = acc[h][e];
    }
    named_bar_sync(1, kConsumerWarps * 32);

    const size_t head0 = static_cast<size_t>(r) * hq + static_cast<size_t>(g) * gsize;
    for (int idx = threadIdx.x; idx < gsize * D; idx += kConsumerWarps * 32) {
        const int h = idx / D, dd = idx % D;
        float o = obuf[h * D + dd];
        for (int ww = 1; ww < kRuns; ++ww) o += obuf[(ww * G + h) * D + dd];
        part[((head0 + h) * cmax + ci) * (D + 4) + 4 + dd] = o;
    }
    if (threadIdx.x < gsize) {
        const int h = threadIdx.x;
        float l = lw[h], mh = mw[h];
        for (int ww = 1; ww < kRuns; ++ww) {
            l += lw[ww * G + h];
            mh = fmaxf(mh, mw[ww * G + h]);
        }
        float* rec = part + ((head0 + h) * cmax + ci) * (D + 4);
        rec[0] = mh;
        rec[1] = l;
    }
}

template <int D>
__global__ void __launch_bounds__(D / 4)
decode_merge_kernel(const float* __restrict__ part, const int32_t* __restrict__ pos, int hq, int win, int ring,
                    int cmax, __nv_bfloat16* __restrict__ out, WsHeader* __restrict__ hdr, int* __restrict__ flags) {
    const int rh = blockIdx.x;
    const int r = rh / hq;
    const int p = checked_pos(pos, r, win, ring, &hdr->status, false);
    const int lo = win > 0 ? max(0, p - win + 1) : 0;
    const int nc = p / kChunk - lo / kChunk + 1;
    const float* rec = part + static_cast<size_t>(rh) * cmax * (D + 4);

    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, rec[c * (D + 4)]);
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    for (int c = 0; c < nc; ++c) {
        const float* rc = rec + c * (D + 4);
        const float ac = expf(rc[0] - M);
        den = fmaf(ac, rc[1], den);
        const float4 o = reinterpret_cast<const float4*>(rc + 4)[threadIdx.x];
        num.x = fmaf(ac, o.x, num.x);
        num.y = fmaf(ac, o.y, num.y);
        num.z = fmaf(ac, o.z, num.z);
        num.w = fmaf(ac, o.w, num.w);
    }
    const float ox = __fdiv_rn(num.x, den), oy = __fdiv_rn(num.y, den);
    const float oz = __fdiv_rn(num.z, den), ow = __fdiv_rn(num.w, den);
    __nv_bfloat162 b01 = __floats2bfloat162_rn(ox, oy);
    __nv_bfloat162 b23 = __floats2bfloat162_rn(oz, ow);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&b01);
    packed.y = *reinterpret_cast<uint32_t*>(&b23);
    reinterpret_cast<uint2*>(out + static_cast<size_t>(rh) * D)[threadIdx.x] = packed;
    const bool bad = !(isfinite(ox) && isfinite(oy) && isfinite(oz) && isfinite(ow));
    if (__syncthreads_or(bad) && threadIdx.x == 0) {
        const int slot = atomicAdd(&hdr->nflag, 1);
        flags[slot] = rh;
    }
}

// [rows, ring, hkv, d] bf16 as a 4-D tensor map with a box of d x 1 x 32 x 1 (no swizzle).
bool encode_ring(CUtensorMap* m, const void* base, int d, int hkv, int ring, int rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(ring),
                          static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(hkv) * d * 2,
                             static_cast<cuuint64_t>(ring) * hkv * d * 2};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(d), 1, static_cast<cuuint32_t>(kRun), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_part(const DecodeArgs& a, cudaStream_t s) {
    using C = PartCfg<D, G>;
    RingMaps maps;
    if (!encode_ring(&maps.tk, a.k, D, a.hkv, a.ring, a.rows) || !encode_ring(&maps.tv, a.v, D, a.hkv, a.ring, a.rows))
        return cudaErrorInvalidValue;
    const dim3 grid(a.cmax, a.hkv, a.rows);
    decode_part_kernel<D, G><<<grid, kPartThreads, C::SMEM, s>>>(
        maps, static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
        static_cast<const __nv_bfloat16*>(a.v), a.pos, a.hq, a.hkv, a.hq / a.hkv, a.win, a.ring, a.scale, a.cmax, a.part,
        &a.hdr->status);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t set_part_attr() {
    return cudaFuncSetAttribute(decode_part_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PartCfg<D, G>::SMEM);
}

template <int D>
cudaError_t prepare_d() {
    cudaError_t e;
    if ((e = set_part_attr<D, 1>()) != cudaSuccess) return e;
    if ((e = set_part_attr<D, 2>()) != cudaSuccess) return e;
    if ((e = set_part_attr<D, 4>()) != cudaSuccess) return e;
    if ((e = set_part_attr<D, 8>()) != cudaSuccess) return e;
    return set_part_attr<D, 16>();
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
    const int G = a.hq / a.hkv;
    cudaError_t e;
    if (G < 1 || G > 16) return cudaErrorInvalidValue;
    if (G >= kTcMinGroup) e = launch_decode_tc_part(a, s);
    else if (G == 1) e = launch_part<D, 1>(a, s);
    else if (G == 2) e = launch_part<D, 2>(a, s);
    else if (G <= 4) e = launch_part<D, 4>(a, s);
    else if (G <= 8) e = launch_part<D, 8>(a, s);
    else e = launch_part<D, 16>(a, s);
    if (e != cudaSuccess) return e;
    decode_merge_kernel<D><<<a.rows * a.hq, D / 4, 0, s>>>(a.part, a.pos, a.hq, a.win, a.ring, a.cmax,
                                                         static_cast<__nv_bfloat16*>(a.out), a.hdr, a.flags);
    return cudaGetLastError();
}

}  // namespace

cudaError_t decode_prepare_device(int dev) {
    cudaError_t e = prepare_d<128>();
    if (e != cudaSuccess) return e;
    if ((e = prepare_d<256>()) != cudaSuccess) return e;
    return decode_tc_prepare_device(dev);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    return a.d == 256 ? launch_d<256>(a, s) : launch_d<128>(a, s);
}

}  // namespace wa
