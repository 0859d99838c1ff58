// wa_static.cu — wa_decode_static: the decode form with a library-owned,
// statically sized workspace, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a plug-in inside a host framework that
// owns all device memory and hands plug-ins no allocator, or a serving loop
// that forbids allocation after start-up because cudaMalloc can synchronize
// the device and stall every stream.  For them this entry point takes the
// same inputs and output as wa_decode but no workspace: the chunk partials,
// the status word and the re-run list live in one file-scope __device__
// array of kStaticWsBytes, which every GPU that loads the library holds until
// the process exits.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "wa.h"
#include "wa_internal.h"

namespace {

constexpr size_t kStaticWsBytes = static_cast<size_t>(WA_STATIC_WS_BYTES);

// The scratch itself.  Host code must not pass this symbol to a kernel: on the
// host it names a stand-in, not device memory.  Its device address comes from
// cudaGetSymbolAddress, looked up once per device in static_ws().
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_ptr[kMaxDevices];
int g_ws_state[kMaxDevices];   // 0 unknown, 1 ready, negative: a WA_E* code

// Once per device, with that device current: capability check, kernel
// attributes, and the device address of g_static_ws.
int static_ws(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WA_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return WA_EDEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_ws_state[dev] < 0) return g_ws_state[dev];
    if (g_ws_state[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return WA_ECUDA;
        if (major != 10 || minor != 3) {
            g_ws_state[dev] = WA_EDEVICE;
            return WA_EDEVICE;
        }
        if (wa::decode_prepare_device(dev) != cudaSuccess) return WA_ECUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return WA_ECUDA;
        g_ws_ptr[dev] = p;
        g_ws_state[dev] = 1;
    }
    *out = g_ws_ptr[dev];
    return WA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace wa {

// The device address of the current device's static array (set up on first use), for wa_status
// with a null workspace: its first 256 bytes are the header the last wa_decode_static call wrote.
int static_ws_header(void** out) { return static_ws(out); }

}  // namespace wa

extern "C" int wa_decode_static(const void* q, const void* k_ring, const void* v_ring, const int32_t* pos,
                                int32_t rows, int32_t hq, int32_t hkv, int32_t d, int32_t win, int32_t ring,
                                float scale, void* out, void* stream) {
    if (!q || !k_ring || !v_ring || !pos || !out) return WA_EINVAL;
    if (rows <= 0 || rows > 65535 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || hq / hkv > 16 || hkv > 65535)
        return WA_EINVAL;
    if (d != 128 && d != 256) return WA_EINVAL;
    if (win < 0 || ring <= 0 || win > ring) return WA_EINVAL;
    if (!std::isfinite(scale)) return WA_EINVAL;
    if (!aligned16(q) || !aligned16(k_ring) || !aligned16(v_ring) || !aligned16(out)) return WA_EINVAL;
    const size_t need = wa_decode_ws_bytes(rows, hq, d, win, ring);
    if (need == 0) return WA_EINVAL;
    if (need > kStaticWsBytes) return WA_ESTATIC;

    void* ws = nullptr;
    const int rc = static_ws(&ws);
    if (rc != WA_OK) return rc;

    // Same layout as a caller-owned workspace: header, re-run list, chunk partials.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    const size_t flags_bytes = (static_cast<size_t>(rows) * hq * sizeof(int) + 255) / 256 * 256;
    wa::DecodeArgs a{};
    a.q = q; a.k = k_ring; a.v = v_ring; a.pos = pos;
    a.rows = rows; a.hq = hq; a.hkv = hkv; a.d = d; a.win = win; a.ring = ring; a.scale = scale;
    a.out = out;
    a.hdr = reinterpret_cast<wa::WsHeader*>(base);
    a.flags = reinterpret_cast<int*>(base + wa::kHeaderBytes);
    a.part = reinterpret_cast<float*>(base + wa::kHeaderBytes + flags_bytes);
    a.cmax = wa::decode_chunks_max(win, ring);
    // The array keeps the previous call's contents: the status word and the
    // re-run counter must start at zero.  The partials are fully rewritten.
    if (cudaMemsetAsync(base, 0, wa::kHeaderBytes, s) != cudaSuccess) return WA_ECUDA;
    if (wa::launch_decode(a, s) != cudaSuccess) return WA_ECUDA;

    wa::RerunArgs r{};
    r.mode = 0; r.q = q; r.k = k_ring; r.v = v_ring; r.idx = pos;
    r.rows = rows; r.hq = hq; r.hkv = hkv; r.d = d; r.win = win; r.ring = ring; r.p0 = 0; r.scale = scale;
    r.out = out; r.hdr = a.hdr; r.flags = a.flags;
    if (wa::launch_rerun(r, s) != cudaSuccess) return WA_ECUDA;
    return WA_OK;
}
