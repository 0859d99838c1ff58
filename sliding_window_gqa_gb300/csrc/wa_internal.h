// wa_internal.h — launch-side structures shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace wa {

constexpr int kChunk = 256;     // decode: keys per chunk, at absolute positions [256c, 256c+255]
constexpr int kHeaderBytes = 256;

// First 256 bytes of every workspace.  The per-call clear resets them.
struct WsHeader {
    int status;   // WA_STATUS_* bits
    int nflag;    // (row, head) pairs queued for the float64 re-run
    int next_unit;   // tensor-core decode: units taken so far past the first one of each CTA
    int pad[61];
};

inline int decode_chunks_max(int win, int ring) {
    return win > 0 ? (win - 1 + kChunk - 1) / kChunk + 1 : (ring + kChunk - 1) / kChunk;
}

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* pos;
    int rows, hq, hkv, d, win, ring;
    float scale;
    void* out;
    WsHeader* hdr;
    int* flags;      // [rows * hq]
    float* part;     // [rows, hq, cmax, d + 4]
    int cmax;
};

struct PromptArgs {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* hi;   // may be null
    int p0, n, hq, hkv, d, win, ring;
    float scale;
    int p32;
    int64_t q_tok, k_tok, v_tok, o_tok;   // token strides, elements
    void* out;
    WsHeader* hdr;
    int* flags;      // [n * hq]
    const int32_t* sel;   // block-sparse form: [n, hkv, nsel] selected 64-key blocks; null otherwise
    int nsel;
};

// Float64 re-run of every flagged (row, head); mode 0 = decode, 1 = prompt, 2 = block-sparse prompt.
struct RerunArgs {
    int mode;
    const int32_t* sel;   // mode 2: [rows, hkv, nsel] selected 64-key blocks
    int nsel;
    const void* q;
    const void* k;
    const void* v;
    const int32_t* idx;  // decode: pos; prompt: hi (may be null)
    int rows, hq, hkv, d, win, ring, p0;
    float scale;
    int64_t q_tok, k_tok, v_tok, o_tok;   // prompt token strides; decode uses dense layouts
    void* out;
    WsHeader* hdr;
    const int* flags;
};

// q/k preparation and KV append (mode WA_PREP_*).
struct PrepArgs {
    const void* src;
    const int32_t* pos;
    const float* q_scale;    // may be null
    const float* inv_freq;   // WA_PREP_L2_ROPE only
    void* q_out;
    void* k_ring;
    void* v_ring;            // may be null
    int n, hq, hkv, d, ring, mode;
    int64_t src_tok, q_tok, ring_row, slot;
    WsHeader* hdr;
};

// cuTensorMapEncodeTiled from the driver, looked up once; null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_prompt(const PromptArgs& a, cudaStream_t s);
cudaError_t launch_prompt_sparse(const PromptArgs& a, cudaStream_t s);
cudaError_t prompt_sparse_prepare_device(int dev);
cudaError_t launch_rerun(const RerunArgs& a, cudaStream_t s);
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);
cudaError_t prompt_prepare_device(int dev);
cudaError_t decode_prepare_device(int dev);
// Decode partials on the tensor cores (query-head groups of kTcMinGroup and more); the merge is shared.
constexpr int kTcMinGroup = 3;
cudaError_t launch_decode_tc_part(const DecodeArgs& a, cudaStream_t s);
cudaError_t decode_tc_prepare_device(int dev);
// Device address of wa_decode_static's scratch on the current device (WA_OK or a WA_E* code).
int static_ws_header(void** out);

}  // namespace wa
