/*
 * wa.h — sliding-window grouped-query attention on one GB300 (sm_103a).
 *
 * Plain C ABI: device pointers, host scalars, one CUDA stream handle passed
 * as void*.  No call allocates, frees or synchronizes, except wa_status,
 * which reads the status word back and therefore waits for the stream.
 *
 * The operation, as defined by TensorFold pull request #1123 ("window_attention
 * at head dim 256"), section "What this changes":
 *
 *   o[row, h] = softmax(scale * q[row, h] . K^T) V  over the row's visible keys,
 *
 * where query head h reads key head g = h / G (G = hq / hkv, at most 16), the
 * key at absolute position j lives in ring slot j mod ring, and the visible
 * keys are [lo, last] with lo = max(0, p - win + 1) for win > 0 and lo = 0 for
 * win = 0 (a linear cache whose ring is its length).  Probabilities stay fp32;
 * the output is bf16, round to nearest even.  Any (row, head) whose output is
 * NaN or infinite is recomputed in float64 (bullet "A NaN or infinite output
 * re-runs its head in float64"), so non-finite outputs carry float64's class.
 *
 * bf16 tensors are passed as raw 16-bit storage (const void*).  Every tensor
 * base pointer must be 16-byte aligned, and every token stride a multiple of
 * 8 elements.  A row's output bits depend only on that row's inputs: not on
 * the batch around it, its slot in the batch, the declared cache length, or
 * how a prompt is cut into chunks.
 *
 * Return codes: WA_OK (0) or a negative WA_E* code.  Argument errors are
 * reported before anything is enqueued.  Errors that only the device can see
 * (a bad pos or hi value in device memory, a wait that ran out) are clamped
 * for memory safety and reported as WA_STATUS_* bits through wa_status.
 */
#ifndef WA_H
#define WA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WA_OK 0
#define WA_EINVAL (-1)        /* an argument is outside the supported set */
#define WA_EWORKSPACE (-2)    /* ws is null, misaligned or smaller than the *_ws_bytes query */
#define WA_ECUDA (-3)         /* a CUDA call or launch failed */
#define WA_EDEVICE (-4)       /* the current device is not a compute capability 10.3 GPU */
#define WA_ESTATIC (-5)       /* wa_decode_static: these sizes need more than WA_STATIC_WS_BYTES of scratch */

/* Size of the library-owned scratch array behind wa_decode_static (16 MiB per device). */
#define WA_STATIC_WS_BYTES (16u * 1024u * 1024u)

#define WA_STATUS_BAD_POS 1   /* a decode pos was < 0, or >= ring with win = 0 (clamped); an append pos < 0 (skipped) */
#define WA_STATUS_BAD_HI 2    /* a prompt hi[i] was outside [p0+i, p0+n-1] (clamped) */
#define WA_STATUS_TIMEOUT 4   /* a bounded device wait gave up; outputs are not valid */
#define WA_STATUS_LAYOUT 8    /* a kernel found its shared memory misaligned and wrote nothing */

/* Token strides in elements for the prompt form (head stride is always d).
 * Zero means dense: hq*d for q and out, hkv*d for k and v. */
typedef struct wa_strides {
    int64_t q;
    int64_t k;
    int64_t v;
    int64_t out;
} wa_strides;

/* Workspace bytes wa_decode needs for these sizes: a 256-byte header (status
 * word, re-run list), one int32 re-run slot per (row, head), and one fp32
 * partial (m, l, o[d]) per (row, head, 256-key chunk).  0 for invalid sizes. */
size_t wa_decode_ws_bytes(int32_t rows, int32_t hq, int32_t d, int32_t win, int32_t ring);

/*
 * Decode form (bullet "Decode" of "What this changes"): few rows, long cache.
 *
 *   q      [rows, hq, d]         bf16, dense
 *   k_ring [rows, ring, hkv, d]  bf16, dense; row r owns ring k_ring[r]
 *   v_ring [rows, ring, hkv, d]  bf16, dense
 *   pos    [rows]                int32, device; row r's last key position p
 *   out    [rows, hq, d]         bf16, written
 *   ws     wa_decode_ws_bytes(...) bytes of device memory, 256-byte aligned
 *
 * Keys are processed in 256-key chunks at absolute positions [256c, 256c+255];
 * one CTA per (chunk, key head, row) writes the chunk's (m, l, o) in fp32, and
 * a second kernel merges the chunks in chunk order:
 * o = sum_c a_c o_c / sum_c a_c l_c with a_c = exp(m_c - M).
 * d is 128 or 256; hq % hkv == 0 and hq / hkv <= 16; 0 <= win <= ring; win = 0
 * needs pos < ring.  Returns WA_EINVAL otherwise.
 */
int wa_decode(const void* q, const void* k_ring, const void* v_ring, const int32_t* pos,
              int32_t rows, int32_t hq, int32_t hkv, int32_t d, int32_t win, int32_t ring,
              float scale, void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * wa_decode_static — wa_decode without a caller workspace.  The pages have no
 * counterpart; it exists for callers that cannot allocate device memory: a
 * plug-in inside a host framework that owns all device memory and gives
 * plug-ins no allocator, or a serving loop that forbids cudaMalloc after
 * start-up because it can synchronize the device and stall every stream.
 *
 * Arguments, layouts and results are those of wa_decode.  The scratch (chunk
 * partials, status word, re-run list) is one library-owned device array of
 * WA_STATIC_WS_BYTES per device, held from library load until process exit;
 * sizes whose wa_decode_ws_bytes exceeds it return WA_ESTATIC before anything
 * is enqueued.  Nothing is allocated or freed.
 *
 * The first call on each device looks up the array's device address (once,
 * with that device current); make that first call before any stream capture.
 * The address is kept for the life of the process: do not call this entry
 * point again after cudaDeviceReset, which unloads the module that holds the
 * array.  Every call on a device shares the one array, and each call clears
 * the status word and re-run counter at its start: calls whose work can
 * overlap on the GPU (for example, calls on two streams with no ordering
 * between them) race on it and must be ordered by the caller; calls on one
 * stream are ordered already.  wa_status(NULL, stream) returns the status
 * bits the last call on the current device left in the array.
 */
int wa_decode_static(const void* q, const void* k_ring, const void* v_ring, const int32_t* pos,
                     int32_t rows, int32_t hq, int32_t hkv, int32_t d, int32_t win, int32_t ring,
                     float scale, void* out, void* stream);

/* Workspace bytes wa_prompt needs: the 256-byte header and one int32 re-run
 * slot per (row, head).  0 for invalid sizes. */
size_t wa_prompt_ws_bytes(int32_t n, int32_t hq);

/*
 * Prompt form (bullets "Prompt", "Window.p32" and "promptRows(..., hi)"):
 * n rows at positions p0 .. p0+n-1 of one sequence.
 *
 *   q    [n, hq, d]      bf16, token stride strides->q (default hq*d)
 *   k    [ring, hkv, d]  bf16, token stride strides->k (default hkv*d); the
 *                        chunk's own keys are already in the ring
 *   v    [ring, hkv, d]  bf16, token stride strides->v (default hkv*d)
 *   hi   [n] int32, device, or NULL: row i sees keys [lo_i, hi[i]] with
 *        p0+i <= hi[i] <= p0+n-1; NULL means hi[i] = p0+i (causal)
 *   p32  0: P enters P.V as one bf16; 1: as bf16(P) + bf16(P - bf16(P))
 *        (bullet "Window.p32"); 2: as three bf16 parts hi + mid + lo whose fp32
 *        sum is P (TensorFold pull request #1622, review thread), which with
 *        the exact bf16 q.k products keeps the result to fp32 accuracy
 *   out  [n, hq, d]      bf16, token stride strides->out (default hq*d)
 *
 * Tensor-core tiles (tcgen05, accumulators in tensor memory, operands staged
 * by TMA) over 128-row query tiles and key tiles at absolute positions, with
 * an fp32 online softmax.  Constraints: d in {128, 256}; hq % hkv == 0 and
 * hq / hkv <= 16; n >= 1, p0 >= 0; for win > 0, win <= ring and the chunk
 * plus its window fits the ring (p0+n-1 - max(0, p0-win+1) < ring); for
 * win = 0, p0 + n <= ring.  Returns WA_EINVAL otherwise.
 */
int wa_prompt(const void* q, const void* k, const void* v, int32_t p0, int32_t n,
              const int32_t* hi, int32_t hq, int32_t hkv, int32_t d, int32_t win, int32_t ring,
              float scale, int32_t p32, const wa_strides* strides, void* out,
              void* ws, size_t ws_bytes, void* stream);

/* Block-sparse prompt: keys per selectable block, and blocks a row may list. */
#define WA_SPARSE_BLOCK 64
#define WA_SPARSE_MAX_SEL 64

/*
 * Block-sparse prompt form (TensorFold pull request #1622, "What this
 * changes": per-row block masks and causal ends over selected key blocks).
 * As wa_prompt, except that row i and query head h (key head g = h / G) see
 * only the keys of [lo_i, hi[i]] whose block j / WA_SPARSE_BLOCK is listed in
 * sel[i, g, 0 .. nsel).  Entries < 0 are unused; repeats and order do not
 * matter.  A row that sees no key gets 0/0 = NaN.
 *
 *   sel   [n, hkv, nsel] int32, device; 1 <= nsel <= WA_SPARSE_MAX_SEL
 *
 * Each CTA takes one key head, its G query heads and 128 / G rows, and runs
 * over the union of those rows' visible selected blocks in key order; a block
 * a row did not select adds nothing to that row, so its bits do not depend on
 * the other rows.  The key span [max(0, p0 - win + 1), p0 + n - 1] may cover
 * at most 65,536 blocks.  Returns WA_EINVAL otherwise, or if sel is NULL.
 */
int wa_prompt_sparse(const void* q, const void* k, const void* v, int32_t p0, int32_t n,
                     const int32_t* hi, int32_t hq, int32_t hkv, int32_t d, int32_t win, int32_t ring,
                     float scale, int32_t p32, const int32_t* sel, int32_t nsel, const wa_strides* strides,
                     void* out, void* ws, size_t ws_bytes, void* stream);

/* Preparations for wa_prep_append. */
#define WA_PREP_RMSNORM 1     /* per-head RMSNorm of q and k */
#define WA_PREP_L2_ROPE 2     /* rotate-half RoPE, L2 norm, q scale */

/* Workspace bytes wa_prep_append needs: the 256-byte header (status word). */
#define WA_PREP_WS_BYTES 256u

/* Layout of wa_prep_append, strides in elements (the head stride is always d). */
typedef struct wa_prep_layout {
    int64_t src_tok;    /* between consecutive tokens' projection rows */
    int64_t q_tok;      /* between consecutive tokens' rows of q_out */
    int64_t ring_row;   /* between the rings of consecutive tokens; 0 = one shared ring */
    int64_t slot;       /* between consecutive slots of a ring */
} wa_prep_layout;

/*
 * q/k preparation and KV append: the step that feeds the caches wa_decode and
 * wa_prompt read.  For each of n tokens, src holds hq query heads, then hkv key
 * heads, then hkv value heads, d bf16 values each (the interleaved projection
 * row of page "Exact Numerical Contract", section "Canonical Boundary").
 *
 *   mode WA_PREP_RMSNORM (page "Exact Numerical Contract", section
 *     "Preparation"): q and k heads become x / sqrt(mean(x^2) + 1e-5),
 *     computed in fp32 and rounded once to bf16 RN.
 *   mode WA_PREP_L2_ROPE (TensorFold pull request #1257, section "What the
 *     kernel computes"): rotate-half RoPE in fp32 (dimension j < d/2 pairs with
 *     j + d/2; angle fl32(pos * inv_freq[j]), fp32 cosf/sinf), rounded to bf16;
 *     then x * (1 / sqrt(sum(x^2) + 1e-6)), rounded to bf16; q heads are then
 *     multiplied by q_scale[j] in fp32 and rounded to bf16.
 *
 *   src      [n] rows of (hq + 2 hkv) * d bf16, token stride lay->src_tok
 *   pos      [n] int32, device: the token's position; a negative position is
 *            reported (WA_STATUS_BAD_POS) and that token is not written
 *   q_scale  [d] fp32, device, or NULL (1.0); WA_PREP_L2_ROPE only
 *   inv_freq [d/2] fp32, device; required for WA_PREP_L2_ROPE, ignored otherwise
 *   q_out    prepared q: token t's head h at q_out + t*q_tok + h*d
 *   k_ring   prepared k: key head g of token t at
 *            k_ring + t*ring_row + (pos[t] mod ring)*slot + g*d
 *   v_ring   v copied as is, same addressing; NULL when v already sits there
 *   ws       WA_PREP_WS_BYTES of device memory, 256-byte aligned (status word)
 *
 * q_out and k_ring may be the very src locations they replace (an in-place
 * preparation of an interleaved buffer, with slot = src_tok and pos[t] = t);
 * any other overlap is undefined.  Constraints: d in {128, 256}; hq % hkv == 0
 * and hq / hkv <= 16; n >= 1; ring >= 1; pointers 16-byte aligned, strides
 * multiples of 8 elements.  Returns WA_EINVAL otherwise.
 */
int wa_prep_append(const void* src, const int32_t* pos, int32_t n, int32_t hq, int32_t hkv, int32_t d,
                   int32_t mode, const float* q_scale, const float* inv_freq, int32_t ring,
                   const wa_prep_layout* lay, void* q_out, void* k_ring, void* v_ring,
                   void* ws, size_t ws_bytes, void* stream);

/* Waits for `stream`, then returns the WA_STATUS_* bits the last call that
 * used `ws` left (0 when clean), or a negative WA_E* code if the read fails.
 * With ws NULL it reads the header of wa_decode_static's scratch array on the
 * current device, i.e. the bits of the last wa_decode_static call there. */
int wa_status(const void* ws, void* stream);

/* Static description of a WA_* return code or WA_STATUS_* bit set. */
const char* wa_strerror(int code);

/* Library version, major * 10000 + minor * 100 + patch. */
int wa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WA_H */
