// wa_rerun.cu — float64 re-run of every (row, head) whose output was NaN or infinite.
//
// TensorFold pull request #1123, section "What this changes", bullet "A NaN
// or infinite output re-runs its head in float64", limited to the affected
// row and head as the review thread settles (the block-wide OR made a finite
// row's bits depend on where a chunk boundary fell).
//
// The block-sparse prompt (mode 2) re-runs over the row's visible keys that lie
// in its selected 64-key blocks (TensorFold pull request #1622); a row with none
// gets 0 / 0 = NaN, as the formula's empty sums give.
//
// A grid of a few CTAs per SM (at most one per (row, head)) walks the flagged
// list; with nothing flagged every CTA exits at once.  Per flagged head:
//   pass 0  fp32 scores (each bf16 x bf16 product is exact in fp32), keys in
//           parallel, 256 at a time.  A key whose fp32 score is not finite is
//           scored again in float64; a float64 score that is NaN or +inf makes
//           the NaN-propagating maximum M NaN or +inf, and then every weight
//           exp(s_j - M) of the formula is NaN or 0 with a NaN sum: the output
//           is NaN, written at once without the float64 passes.  (A NaN key
//           seen by many rows flags every one of them; this settles them
//           without float64 dot products over the whole window.)
//   pass 1  the float64 NaN-propagating maximum score M;
//   pass 2  w_j = exp(s_j - M) block by block and sum_j w_j v_j in key order,
//           one thread per output dim.
// Key j always goes to thread (j - lo) mod 256 and the reductions use fixed
// trees, so the bits depend only on the row's own inputs.
#include <cuda_bf16.h>

#include "wa_internal.h"
#include "wa_ptx.cuh"

namespace wa {

namespace {

constexpr int kRerunThreads = 256;

__device__ __forceinline__ double bf16_bits_to_f64(uint16_t b) {
    return static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16));
}

// Round a float64 value to bf16, nearest-even, in one step; an underflow keeps its sign.
__device__ uint16_t f64_to_bf16_rn(double x) {
    const uint16_t sign = (__double_as_longlong(x) < 0) ? 0x8000u : 0u;
    if (isnan(x)) return sign | 0x7FC0u;
    const double ax = fabs(x);
    if (isinf(ax)) return sign | 0x7F80u;
    if (ax < 0x1p-126) {   // subnormal range: quantum 2^-133
        return sign | static_cast<uint16_t>(rint(ax * 0x1p133));
    }
    int e;
    const double m = frexp(ax, &e);      // ax = m * 2^e, m in [0.5, 1)
    double sig = rint(ldexp(m, 8));      // 8 significant bits
    if (sig >= 256.0) {
        sig = 128.0;
        e += 1;
    }
    const int biased = e - 1 + 127;
    if (biased >= 255) return sign | 0x7F80u;
    return sign | static_cast<uint16_t>((biased << 7) | (static_cast<int>(sig) - 128));
}

__device__ __forceinline__ double block_reduce(double x, bool is_max, double* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const double y = __shfl_xor_sync(0xFFFFFFFFu, x, off);
        x = is_max ? ((isnan(x) || isnan(y)) ? (x + y) : fmax(x, y)) : (x + y);
    }
    if (lane == 0) red[warp] = x;
    __syncthreads();
    double r = red[0];
    for (int w = 1; w < kRerunThreads / 32; ++w) {
        const double y = red[w];
        r = is_max ? ((isnan(r) || isnan(y)) ? (r + y) : fmax(r, y)) : (r + y);
    }
    __syncthreads();
    return r;
}

// d bf16 values of a row as float64 (16-byte loads; the row is 16-byte aligned).
__device__ __forceinline__ double dot_f64(const double* qd, const uint16_t* kr, int d) {
    double s = 0.0;
    for (int e = 0; e < d; e += 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(kr + e);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s = s + qd[e + 2 * i] * static_cast<double>(__uint_as_float(w[i] << 16));
            s = s + qd[e + 2 * i + 1] * static_cast<double>(__uint_as_float(w[i] & 0xFFFF0000u));
        }
    }
    return s;
}

// The same dot product in fp32: every product of two bf16 values is exact in fp32 unless it
// overflows or underflows, so a finite float64 score can only come out non-finite here through
// overflow, and a float64 NaN or infinity always shows as non-finite.
__device__ __forceinline__ float dot_f32(const float* qf, const uint16_t* kr, int d) {
    float s = 0.f;
    for (int e = 0; e < d; e += 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(kr + e);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s = fmaf(qf[e + 2 * i], __uint_as_float(w[i] << 16), s);
            s = fmaf(qf[e + 2 * i + 1], __uint_as_float(w[i] & 0xFFFF0000u), s);
        }
    }
    return s;
}

__global__ void __launch_bounds__(kRerunThreads) rerun_f64_kernel(RerunArgs a) {
    __shared__ double qd[256];
    __shared__ float qf[256];
    __shared__ double wb[kRerunThreads];
    __shared__ double red[kRerunThreads / 32];
    __shared__ int sel_row[64];
    __shared__ unsigned char vis[kRerunThreads];
    const int nflag = *reinterpret_cast<volatile int*>(&a.hdr->nflag);
    const int t = threadIdx.x;
    const int G = a.hq / a.hkv;
    const int d = a.d;
    const uint16_t* q = static_cast<const uint16_t*>(a.q);
    const uint16_t* k = static_cast<const uint16_t*>(a.k);
    const uint16_t* v = static_cast<const uint16_t*>(a.v);
    uint16_t* out = static_cast<uint16_t*>(a.out);

    for (int f = blockIdx.x; f < nflag; f += gridDim.x) {
        const int rh = a.flags[f];
        const int row = rh / a.hq, h = rh % a.hq, g = h / G;
        int lo, last;
        const uint16_t *qrow, *kb, *vb;
        int64_t kst, vst;
        uint16_t* orow;
        if (a.mode == 0) {
            int p = a.idx[row];
            if (p < 0) p = 0;
            if (a.win == 0 && p >= a.ring) p = a.ring - 1;
            lo = a.win > 0 ? max(0, p - a.win + 1) : 0;
            last = p;
            qrow = q + (static_cast<int64_t>(row) * a.hq + h) * d;
            kb = k + static_cast<int64_t>(row) * a.ring * a.hkv * d + static_cast<int64_t>(g) * d;
            vb = v + static_cast<int64_t>(row) * a.ring * a.hkv * d + static_cast<int64_t>(g) * d;
            kst = vst = static_cast<int64_t>(a.hkv) * d;
            orow = out + (static_cast<int64_t>(row) * a.hq + h) * d;
        } else {
            const int P = a.p0 + row;
            last = P;
            if (a.idx) last = min(max(a.idx[row], P), a.p0 + a.rows - 1);
            lo = a.win > 0 ? max(0, P - a.win + 1) : 0;
            qrow = q + row * a.q_tok + static_cast<int64_t>(h) * d;
            kb = k + static_cast<int64_t>(g) * d;
            vb = v + static_cast<int64_t>(g) * d;
            kst = a.k_tok;
            vst = a.v_tok;
            orow = out + row * a.o_tok + static_cast<int64_t>(h) * d;
        }
        if (t < d) {
            const float x = __uint_as_float(static_cast<uint32_t>(qrow[t]) << 16);
            qf[t] = x * a.scale;   // the scale applied to fp32 q: only the class of the score matters here
            qd[t] = static_cast<double>(x);
        }
        const int nsel = a.mode == 2 ? a.nsel : 0;
        if (t < nsel) sel_row[t] = a.sel[(static_cast<int64_t>(row) * a.hkv + g) * a.nsel + t];
        __syncthreads();
        // mode 2: key j counts only if its block j / 64 is selected
        auto selected = [&](int j) {
            if (a.mode != 2) return true;
            bool hit = false;
            for (int e = 0; e < nsel; ++e) hit |= sel_row[e] == (j >> 6);
            return hit;
        };
        auto score = [&](int j) {
            const uint16_t* kr = kb + static_cast<int64_t>(j % a.ring) * kst;
            return dot_f64(qd, kr, d) * static_cast<double>(a.scale);
        };

        // pass 0: a float64 score that is NaN or +inf makes the output NaN
        bool nan_out = false;
        for (int base = lo; base <= last && !nan_out; base += kRerunThreads) {
            const int j = base + t;
            bool hit = false;
            if (j <= last && selected(j)) {
                const float sf = dot_f32(qf, kb + static_cast<int64_t>(j % a.ring) * kst, d);
                if (!isfinite(sf)) {
                    const double s = score(j);
                    hit = isnan(s) || (isinf(s) && s > 0.0);
                }
            }
            nan_out = __syncthreads_or(hit) != 0;
        }
        if (nan_out) {
            if (t < d) orow[t] = 0x7FC0u;
            __syncthreads();
            continue;
        }

        // pass 1: the maximum score (NaN if any score is NaN)
        double mloc = -INFINITY;
        for (int j = lo + t; j <= last; j += kRerunThreads) {
            if (!selected(j)) continue;
            const double s = score(j);
            mloc = (isnan(s) || isnan(mloc)) ? (s + mloc) : fmax(mloc, s);
        }
        const double M = block_reduce(mloc, true, red);

        // pass 2: weights, their sum, and sum_j w_j v_j in key order
        double lloc = 0.0, acc = 0.0;
        for (int base = lo; base <= last; base += kRerunThreads) {
            const int j = base + t;
            double w = 0.0;
            const bool use = j <= last && selected(j);
            if (use) {
                w = exp(score(j) - M);
                lloc = lloc + w;
            }
            wb[t] = w;
            vis[t] = use ? 1 : 0;
            __syncthreads();
            if (t < d) {
                const int cnt = min(kRerunThreads, last - base + 1);
                for (int jj = 0; jj < cnt; ++jj)
                    if (vis[jj])
                        acc = acc + wb[jj] * bf16_bits_to_f64(vb[static_cast<int64_t>((base + jj) % a.ring) * vst + t]);
            }
            __syncthreads();
        }
        const double l = block_reduce(lloc, false, red);
        if (t < d) orow[t] = f64_to_bf16_rn(acc / l);
        __syncthreads();
    }
}

}  // namespace

// A few CTAs per SM, never more than the (row, head) pairs that can be flagged: the grid is
// fixed before the flag count is known (no host read), and CTAs past the count exit at once.
cudaError_t launch_rerun(const RerunArgs& a, cudaStream_t s) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    const int64_t units = static_cast<int64_t>(a.rows) * a.hq;
    const int grid = static_cast<int>(units < 4LL * sms ? units : 4LL * sms);
    rerun_f64_kernel<<<grid, kRerunThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace wa
