// wa_api.cu — the C ABI: argument checks, workspace carving, launches.
//
// Entry points and their arguments follow the operator of TensorFold pull
// request #1123, section "What this changes": decode (bullet "Decode") and
// prompt rows with an optional per-row last key (bullet "promptRows(...,
// hi)"), a scale parameter and window 0 as a linear cache (bullet "Scale is
// a parameter"), and the optional two-half P (bullet "Window.p32").
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "wa.h"
#include "wa_internal.h"

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_ready[kMaxDevices];   // 0 unknown, 1 ready, negative: a WA_E* code

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool heads_ok(int32_t hq, int32_t hkv) {
    return hq > 0 && hkv > 0 && hq % hkv == 0 && hq / hkv <= 16;
}

// Once per device: capability check and kernel attributes.
int ensure_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WA_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return WA_EDEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_ready[dev] != 0) return g_ready[dev] > 0 ? WA_OK : g_ready[dev];
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return WA_ECUDA;
    if (major != 10 || minor != 3) {
        g_ready[dev] = WA_EDEVICE;
        return WA_EDEVICE;
    }
    if (wa::decode_prepare_device(dev) != cudaSuccess || wa::prompt_prepare_device(dev) != cudaSuccess ||
        wa::prompt_sparse_prepare_device(dev) != cudaSuccess)
        return WA_ECUDA;
    g_ready[dev] = 1;
    return WA_OK;
}

size_t flags_bytes(int64_t units) { return round_up(static_cast<size_t>(units) * sizeof(int), 256); }

}  // namespace

extern "C" {

size_t wa_decode_ws_bytes(int32_t rows, int32_t hq, int32_t d, int32_t win, int32_t ring) {
    if (rows <= 0 || hq <= 0 || (d != 128 && d != 256) || win < 0 || ring <= 0 || win > ring) return 0;
    const int64_t units = static_cast<int64_t>(rows) * hq;
    const int cmax = wa::decode_chunks_max(win, ring);
    return wa::kHeaderBytes + flags_bytes(units) +
           static_cast<size_t>(units) * cmax * static_cast<size_t>(d + 4) * sizeof(float);
}

int wa_decode(const void* q, const void* k_ring, const void* v_ring, const int32_t* pos,
              int32_t rows, int32_t hq, int32_t hkv, int32_t d, int32_t win, int32_t ring,
              float scale, void* out, void* ws, size_t ws_bytes, void* stream) {
    if (!q || !k_ring || !v_ring || !pos || !out) return WA_EINVAL;
    if (rows <= 0 || rows > 65535 || !heads_ok(hq, hkv) || hkv > 65535) return WA_EINVAL;
    if (d != 128 && d != 256) return WA_EINVAL;
    if (win < 0 || ring <= 0 || win > ring) return WA_EINVAL;
    if (!std::isfinite(scale)) return WA_EINVAL;
    if (!aligned16(q) || !aligned16(k_ring) || !aligned16(v_ring) || !aligned16(out)) return WA_EINVAL;
    const size_t need = wa_decode_ws_bytes(rows, hq, d, win, ring);
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return WA_EWORKSPACE;
    const int rc = ensure_device();
    if (rc != WA_OK) return rc;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    wa::DecodeArgs a{};
    a.q = q; a.k = k_ring; a.v = v_ring; a.pos = pos;
    a.rows = rows; a.hq = hq; a.hkv = hkv; a.d = d; a.win = win; a.ring = ring; a.scale = scale;
    a.out = out;
    a.hdr = reinterpret_cast<wa::WsHeader*>(base);
    a.flags = reinterpret_cast<int*>(base + wa::kHeaderBytes);
    a.part = reinterpret_cast<float*>(base + wa::kHeaderBytes + flags_bytes(static_cast<int64_t>(rows) * hq));
    a.cmax = wa::decode_chunks_max(win, ring);
    if (cudaMemsetAsync(base, 0, wa::kHeaderBytes, s) != cudaSuccess) return WA_ECUDA;
    if (wa::launch_decode(a, s) != cudaSuccess) return WA_ECUDA;

    wa::RerunArgs r{};
    r.mode = 0; r.q = q; r.k = k_ring; r.v = v_ring; r.idx = pos;
    r.rows = rows; r.hq = hq; r.hkv = hkv; r.d = d; r.win = win; r.ring = ring; r.p0 = 0; r.scale = scale;
    r.out = out; r.hdr = a.hdr; r.flags = a.flags;
    if (wa::launch_rerun(r, s) != cudaSuccess) return WA_ECUDA;
    return WA_OK;
}

size_t wa_prompt_ws_bytes(int32_t n, int32_t hq) {
    if (n <= 0 || hq <= 0) return 0;
    return wa::kHeaderBytes + flags_bytes(static_cast<int64_t>(n) * hq);
}

}  // extern "C"

namespace {

// wa_prompt and wa_prompt_sparse: shared checks, workspace carving, launch and re-run.
int prompt_call(const void* q, const void* k, const void* v, int32_t p0, int32_t n, const int32_t* hi, int32_t hq,
                int32_t hkv, int32_t d, int32_t win, int32_t ring, float scale, int32_t p32, const int32_t* sel,
                int32_t nsel, const wa_strides* strides, void* out, void* ws, size_t ws_bytes, void* stream) {
    if (!q || !k || !v || !out) return WA_EINVAL;
    if (n <= 0 || p0 < 0 || !heads_ok(hq, hkv) || hq > 65535) return WA_EINVAL;
    if (d != 128 && d != 256) return WA_EINVAL;
    if (win < 0 || ring <= 0 || win > ring) return WA_EINVAL;
    if (p32 < 0 || p32 > 2) return WA_EINVAL;
    if (!std::isfinite(scale)) return WA_EINVAL;
    if (static_cast<int64_t>(p0) + n > INT32_MAX) return WA_EINVAL;
    const int64_t span_lo = win > 0 && p0 - win + 1 > 0 ? p0 - win + 1 : 0;
    if (win > 0) {
        if (static_cast<int64_t>(p0) + n - 1 - span_lo >= ring) return WA_EINVAL;
    } else if (static_cast<int64_t>(p0) + n > ring) {
        return WA_EINVAL;
    }
    if (sel) {
        if (nsel < 1 || nsel > WA_SPARSE_MAX_SEL) return WA_EINVAL;
        // the kernel's union bitmap covers at most 65,536 blocks of the key span
        if ((static_cast<int64_t>(p0) + n - 1) / WA_SPARSE_BLOCK - span_lo / WA_SPARSE_BLOCK + 1 > 65536)
            return WA_EINVAL;
    }
    int64_t qs = static_cast<int64_t>(hq) * d, ks = static_cast<int64_t>(hkv) * d, vs = ks, os = qs;
    if (strides) {
        if (strides->q) qs = strides->q;
        if (strides->k) ks = strides->k;
        if (strides->v) vs = strides->v;
        if (strides->out) os = strides->out;
    }
    if (qs < static_cast<int64_t>(hq) * d || ks < static_cast<int64_t>(hkv) * d || vs < static_cast<int64_t>(hkv) * d ||
        os < static_cast<int64_t>(hq) * d)
        return WA_EINVAL;
    if ((qs | ks | vs | os) & 7) return WA_EINVAL;   // 16-byte token strides (TMA)
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return WA_EINVAL;
    const size_t need = wa_prompt_ws_bytes(n, hq);
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return WA_EWORKSPACE;
    const int rc = ensure_device();
    if (rc != WA_OK) return rc;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    wa::PromptArgs a{};
    a.q = q; a.k = k; a.v = v; a.hi = hi;
    a.p0 = p0; a.n = n; a.hq = hq; a.hkv = hkv; a.d = d; a.win = win; a.ring = ring; a.scale = scale; a.p32 = p32;
    a.q_tok = qs; a.k_tok = ks; a.v_tok = vs; a.o_tok = os;
    a.out = out;
    a.hdr = reinterpret_cast<wa::WsHeader*>(base);
    a.flags = reinterpret_cast<int*>(base + wa::kHeaderBytes);
    a.sel = sel;
    a.nsel = sel ? nsel : 0;
    if (cudaMemsetAsync(base, 0, wa::kHeaderBytes, s) != cudaSuccess) return WA_ECUDA;
    const cudaError_t e = sel ? wa::launch_prompt_sparse(a, s) : wa::launch_prompt(a, s);
    if (e == cudaErrorNotSupported) return WA_EINVAL;
    if (e != cudaSuccess) return WA_ECUDA;

    wa::RerunArgs r{};
    r.mode = sel ? 2 : 1; r.q = q; r.k = k; r.v = v; r.idx = hi;
    r.sel = sel; r.nsel = a.nsel;
    r.rows = n; r.hq = hq; r.hkv = hkv; r.d = d; r.win = win; r.ring = ring; r.p0 = p0; r.scale = scale;
    r.q_tok = qs; r.k_tok = ks; r.v_tok = vs; r.o_tok = os;
    r.out = out; r.hdr = a.hdr; r.flags = a.flags;
    if (wa::launch_rerun(r, s) != cudaSuccess) return WA_ECUDA;
    return WA_OK;
}

}  // namespace

extern "C" {

int wa_prompt(const void* q, const void* k, const void* v, int32_t p0, int32_t n,
              const int32_t* hi, int32_t hq, int32_t hkv, int32_t d, int32_t win, int32_t ring,
              float scale, int32_t p32, const wa_strides* strides, void* out,
              void* ws, size_t ws_bytes, void* stream) {
    return prompt_call(q, k, v, p0, n, hi, hq, hkv, d, win, ring, scale, p32, nullptr, 0, strides, out, ws, ws_bytes,
                       stream);
}

int wa_prompt_sparse(const void* q, const void* k, const void* v, int32_t p0, int32_t n,
                     const int32_t* hi, int32_t hq, int32_t hkv, int32_t d, int32_t win, int32_t ring,
                     float scale, int32_t p32, const int32_t* sel, int32_t nsel, const wa_strides* strides,
                     void* out, void* ws, size_t ws_bytes, void* stream) {
    if (!sel) return WA_EINVAL;
    return prompt_call(q, k, v, p0, n, hi, hq, hkv, d, win, ring, scale, p32, sel, nsel, strides, out, ws, ws_bytes,
                       stream);
}

int wa_prep_append(const void* src, const int32_t* pos, int32_t n, int32_t hq, int32_t hkv, int32_t d,
                   int32_t mode, const float* q_scale, const float* inv_freq, int32_t ring,
                   const wa_prep_layout* lay, void* q_out, void* k_ring, void* v_ring,
                   void* ws, size_t ws_bytes, void* stream) {
    if (!src || !pos || !lay || !q_out || !k_ring) return WA_EINVAL;
    if (n <= 0 || !heads_ok(hq, hkv) || ring <= 0) return WA_EINVAL;
    if (d != 128 && d != 256) return WA_EINVAL;
    if (mode != WA_PREP_RMSNORM && mode != WA_PREP_L2_ROPE) return WA_EINVAL;
    if (mode == WA_PREP_L2_ROPE && !inv_freq) return WA_EINVAL;
    if (!aligned16(src) || !aligned16(q_out) || !aligned16(k_ring) || (v_ring && !aligned16(v_ring))) return WA_EINVAL;
    if (lay->src_tok < (hq + 2 * hkv) * static_cast<int64_t>(d) || lay->q_tok < hq * static_cast<int64_t>(d) ||
        lay->ring_row < 0 || lay->slot < hkv * static_cast<int64_t>(d))
        return WA_EINVAL;
    if ((lay->src_tok | lay->q_tok | lay->ring_row | lay->slot) & 7) return WA_EINVAL;
    if (!ws || ws_bytes < WA_PREP_WS_BYTES || (reinterpret_cast<uintptr_t>(ws) & 255u)) return WA_EWORKSPACE;
    const int rc = ensure_device();
    if (rc != WA_OK) return rc;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    wa::PrepArgs a{};
    a.src = src; a.pos = pos; a.q_scale = mode == WA_PREP_L2_ROPE ? q_scale : nullptr; a.inv_freq = inv_freq;
    a.q_out = q_out; a.k_ring = k_ring; a.v_ring = v_ring;
    a.n = n; a.hq = hq; a.hkv = hkv; a.d = d; a.ring = ring; a.mode = mode;
    a.src_tok = lay->src_tok; a.q_tok = lay->q_tok; a.ring_row = lay->ring_row; a.slot = lay->slot;
    a.hdr = static_cast<wa::WsHeader*>(ws);
    if (cudaMemsetAsync(ws, 0, wa::kHeaderBytes, s) != cudaSuccess) return WA_ECUDA;
    if (wa::launch_prep(a, s) != cudaSuccess) return WA_ECUDA;
    return WA_OK;
}

int wa_status(const void* ws, void* stream) {
    if (!ws) {   // the header of wa_decode_static's scratch on the current device
        void* sws = nullptr;
        const int rc = wa::static_ws_header(&sws);
        if (rc != WA_OK) return rc;
        ws = sws;
    }
    int st = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&st, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return WA_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return WA_ECUDA;
    return st;
}

const char* wa_strerror(int code) {
    switch (code) {
        case WA_OK: return "ok";
        case WA_EINVAL: return "invalid argument";
        case WA_EWORKSPACE: return "workspace missing, misaligned or too small";
        case WA_ECUDA: return "CUDA call or launch failed";
        case WA_EDEVICE: return "device is not compute capability 10.3 (GB300)";
        case WA_ESTATIC: return "sizes need more scratch than wa_decode_static's fixed 16 MiB array";
        case WA_STATUS_BAD_POS: return "status: a decode or append position was out of range (clamped or skipped)";
        case WA_STATUS_BAD_HI: return "status: a prompt hi[i] was out of range (clamped)";
        case WA_STATUS_TIMEOUT: return "status: a device wait ran out; outputs are not valid";
        case WA_STATUS_LAYOUT: return "status: shared memory misaligned; outputs were not written";
        default:
            if (code > 0) return "status: several WA_STATUS bits";
            return "unknown code";
    }
}

int wa_version(void) { return 100; }

}  // extern "C"
