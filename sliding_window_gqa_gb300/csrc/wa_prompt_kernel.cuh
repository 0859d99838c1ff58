// wa_prompt_kernel.cuh — the prompt kernel, shared by the dense and block-sparse forms.
//
// TensorFold pull request #1123 ("window_attention at head dim 256"),
// section "What this changes": bullets "Prompt" (tensor-core tiles, key
// tiles at absolute positions, each folded into o once, so a row's bits do
// not depend on how the prompt is chunked), "Window.p32" (P enters P.V as
// bf16(P) + bf16(P - bf16(P))), "promptRows(..., hi)" (row i sees keys
// [p0 + i - win + 1, hi[i]]) and "Scale is a parameter" (window 0 = linear
// cache).  Probabilities are fp32; the running softmax is fp32.  A third
// P mode carries P as three bf16 parts (hi, mid, lo) whose fp32 sum is P, one
// P.V product per part (TensorFold pull request #1622, review thread: q*scale
// and P "each carried as three 16-bit parts ... with one matrix op per part").
// Here q enters S unscaled and exact, and the scale is applied to S in fp32,
// so only P needs the split; S and the three-part P.V are then accurate to
// fp32.
//
// GB300 design (one CTA per 128-row query tile of one query head):
//   warp 0      TMA producer: Q once, then K and V tiles of T keys into two
//               stages each (128-byte swizzle); tiles that wrap around the
//               ring are copied by the warp with the same swizzle.
//   warp 1      allocates tensor memory; lane 0 issues tcgen05.mma:
//               S = Q K^T into one of two S buffers, then O += P V.
//   warp 2      zeroes V rows outside the CTA's key union in the first and
//               last tile, so stale ring slots never meet a zero P as 0 * inf.
//   warps 4..7  one query row per thread (= tensor-memory lane): mask, scale,
//               online softmax with a lazy rescale, P (bf16) to tensor memory
//               as the A operand of P V, O rescale in tensor memory, epilogue.
// Every mbarrier has one waiter role that takes its phases in order.
//
// Block-sparse form (TensorFold pull request #1622, "What this changes": the
// kv head's query heads over the union of the rows' selected blocks, with
// per-row block masks and causal ends).  A CTA takes one key head and its G
// query heads for R = 128 / G rows: tensor-memory lane m is row m / G, query
// head m % G (lanes from R G on idle), loaded by one TMA box of 64 dims x G
// heads x R rows.  The key tiles are the
// 64-key blocks that any row of the CTA selected and can see, in ascending key
// order (a bitmap over the CTA's key span); each row keeps its sorted block list
// and masks whole the blocks it did not select, so a row's sums are those of its
// own blocks in key order whatever its neighbours selected.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "wa_internal.h"
#include "wa_ptx.cuh"

namespace wa {

namespace {

constexpr int kBM = 128;           // query rows per CTA (= tensor-memory lanes)
constexpr int kThreads = 384;      // warps 0..3 control, 4..7 and 8..11 softmax (two column halves)
constexpr float kLazy = 8.0f;      // log2 units the running max may trail before O is rescaled

struct PromptParams {
    CUtensorMap tq, tk, tv;
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* hi;
    uint16_t* out;
    int* status;
    int* nflag;
    int* flags;
    int64_t k_tok, v_tok, o_tok;
    int p0, n, hq, hkv, win, ring, nqt;
    float c;          // |scale| * log2(e)
    int neg;          // scale < 0: the S MMA negates Q
    // block-sparse form only
    const int32_t* sel;   // [n, hkv, nsel] selected 64-key blocks, -1 = unused
    int nsel;
    int gsz;              // query heads per CTA row: lane m = (row m / gsz, head m % gsz); 1 for dense
    int hfirst;           // CTAs in launch order take every head of one query tile before the next tile
};

constexpr int kSelMax = 64;        // block-sparse: selected blocks per row at most
constexpr int kBitmapWords = 2048; // block-sparse: the CTA's key span in 64-key blocks, at most 65,536

// NP: the parts P enters P.V as (1: bf16(P); 2: hi, lo; 3: hi, mid, lo).
// SP: block-sparse form (tiles are the selected 64-key blocks of the CTA's rows).
template <int D, int NP, bool SP = false>
struct Cfg {
    static constexpr int T = (D == 256 || NP == 3 || SP) ? 64 : 128;   // keys per tile
    static constexpr int NC = T / 2;                  // S columns per softmax thread
    static constexpr int KB = D / 64;                 // 64-element (128-byte) column blocks
    static constexpr int Q_BLOCK = kBM * 128;
    static constexpr int Q_BYTES = KB * Q_BLOCK;
    static constexpr int KV_BLOCK = T * 128;
    static constexpr int KV_BYTES = KB * KV_BLOCK;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;               // 2 stages
    static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;          // 2 stages
    // P lives in tensor memory (the A operand of P.V): two buffers (tiles alternate) for a
    // single bf16 P, one buffer of NP parts otherwise; T / 2 columns each.
    static constexpr int P_BUFS = NP == 1 ? 2 : 1;
    static constexpr int P_SLOTS = NP == 1 ? 2 : NP;
    static constexpr int OFF_X = OFF_V + 2 * KV_BYTES;          // row exchange [2 tiles][2 halves][128] fp32
    static constexpr int OFF_BAR = OFF_X + 2 * 2 * kBM * 4;
    static constexpr int NBAR = 24;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;         // tmem base, union bounds
    // block-sparse: union bitmap over the CTA's key span, each row's sorted block list and count
    static constexpr int OFF_BMAP = OFF_MISC + 64;
    static constexpr int OFF_SEL = OFF_BMAP + (SP ? kBitmapWords * 4 : 0);
    static constexpr int OFF_CNT = OFF_SEL + (SP ? kBM * kSelMax * 2 : 0);
    static constexpr int SMEM = OFF_CNT + (SP ? kBM * 4 : 0);
    static constexpr int TMEM_COLS = 512;
    static constexpr int O_COL = 0;
    static constexpr int S_COL = D;                             // S buffers at D and D + T
    static constexpr int P_COL = D + 2 * T;                     // P: P_SLOTS x T/2 columns
    __host__ __device__ static constexpr int p_col(int buf_or_part) { return P_COL + buf_or_part * (T / 2); }
    static_assert(P_COL + P_SLOTS * (T / 2) <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// barrier indices
enum : int {
    B_Q = 0, B_KFULL = 1, B_VFULL = 3, B_VREADY = 5, B_KFREE = 7, B_VFREE = 9, B_SFULL = 11, B_SFREE = 13,
    B_PFULL = 15, B_PVDONE = 17, B_DRAIN = 19, B_XCHG = 20, B_EPI_L = 22, B_EPI_B = 23   // PFULL, PVDONE: [tile & 1]
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max of three fp32 values in one instruction (a NaN input is passed over, as by fmaxf).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Two fp32 fused multiply-adds (d = a * b + c, round to nearest) in one packed instruction.
__device__ __forceinline__ void fma_x2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                       float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// Two fp32 additions (round to nearest) in one packed instruction: (s0, s1) += (a0, a1).
__device__ __forceinline__ void add_x2(float& s0, float& s1, float a0, float a1) {
    asm("{\n\t.reg .b64 ra, rs;\n\t"
        "mov.b64 rs, {%0, %1};\n\tmov.b64 ra, {%2, %3};\n\t"
        "add.rn.f32x2 rs, rs, ra;\n\tmov.b64 {%0, %1}, rs;\n\t}"
        : "+f"(s0), "+f"(s1) : "f"(a0), "f"(a1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Copy one tile of T key rows (slots (key0 + k) mod ring) into a swizzled stage, by one warp.
// Used for tiles that wrap around the end of the ring, which one TMA box cannot express.
template <int D, int T>
__device__ void copy_tile_wrapped(uint32_t dst, const uint16_t* base, int64_t tok, int g, int key0, int ring,
                                  int lane) {
    constexpr int KB = D / 64;
    constexpr int UNITS = T * KB * 8;   // 16-byte units
    for (int u = lane; u < UNITS; u += 32) {
        const int k = u / (KB * 8);
        const int rem = u % (KB * 8);
        const int b = rem / 8, c = rem % 8;
        const int slot = (key0 + k) % ring;
        const uint4 val = ld_global_nc_v4(base + slot * tok + static_cast<int64_t>(g) * D + b * 64 + c * 8);
        st_shared_v4(dst + b * (T * 128) + k * 128 + ((c ^ (k & 7)) * 16), val.x, val.y, val.z, val.w);
    }
    fence_proxy_async_smem();
}

// The NC S values of this thread's half row: raw fp32 bits from tensor memory.
template <int NC>
__device__ __forceinline__ void load_s(uint32_t taddr, float (&sv)[NC]) {
    if constexpr (NC == 64) {
        uint32_t raw[64];
        tmem_ld64_wait(taddr, raw);
#pragma unroll
        for (int e = 0; e < 64; ++e) sv[e] = __uint_as_float(raw[e]);
    } else {
        uint32_t raw[32];
        tmem_ld32_wait(taddr, raw);
#pragma unroll
        for (int e = 0; e < 32; ++e) sv[e] = __uint_as_float(raw[e]);
    }
}

// Block-sparse: one row's selected blocks that hold a visible key ([blo, bhi]), relative to j0,
// sorted and without repeats, into lst; each also set in the CTA's union bitmap.  All N entries
// are loaded first (unused ones as 0xFFFF, which sorts last), then an ascending bitonic network in
// registers with compile-time indices; N is the smallest of 32 and 64 that holds the row's list.
template <int N>
__device__ __forceinline__ int build_block_list(const int32_t* srow, int nsel, int blo, int bhi, int j0,
                                                uint16_t* lst, uint32_t* bmap) {
    uint32_t v[N];
#pragma unroll
    for (int e = 0; e < N; ++e) {
        const int b = e < nsel ? srow[e] : -1;
        v[e] = (b >= blo && b <= bhi) ? static_cast<uint32_t>(b - j0) : 0xFFFFu;
    }
#pragma unroll
    for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int e = 0; e < N; ++e) {
                const int l = e ^ j;
                if (l > e) {
                    const uint32_t lo = min(v[e], v[l]), hi = max(v[e], v[l]);
                    const bool up = (e & k) == 0;
                    v[e] = up ? lo : hi;
                    v[l] = up ? hi : lo;
                }
            }
        }
    }
    int cnt = 0;
    uint32_t prev = 0xFFFFFFFFu;
#pragma unroll
    for (int e = 0; e < N; ++e) {
        const uint32_t x = v[e];
        if (x != 0xFFFFu && x != prev) {
            lst[cnt++] = static_cast<uint16_t>(x);
            atomicOr(&bmap[x >> 5], 1u << (x & 31));
        }
        prev = x;
    }
    return cnt;
}

// Tiles in ascending key order: the dense form walks j0, j0 + 1, ...; the block-sparse form walks
// the set bits of the CTA's union bitmap.  next() returns the tile's block relative to j0 and is
// called exactly once per tile.
template <bool SP>
struct TileWalk {
    const uint32_t* bm;
    int nw, w, k;
    uint32_t cur;
    __device__ __forceinline__ void init(const uint32_t* bitmap, int nwords) {
        bm = bitmap; nw = nwords; w = 0; k = 0;
        cur = SP ? bitmap[0] : 0u;
    }
    __device__ __forceinline__ int next() {
        if constexpr (!SP) {
            return k++;
        } else {
            while (cur == 0u && w + 1 < nw) cur = bm[++w];
            const int b = __ffs(cur) - 1;
            cur &= cur - 1u;
            return (w << 5) + b;
        }
    }
};

template <int D, int NP, bool SP>
__global__ void __launch_bounds__(kThreads, 1) prompt_kernel(const __grid_constant__ PromptParams p) {
    using C = Cfg<D, NP, SP>;
    constexpr int T = C::T;
    constexpr int NC = C::NC;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {   // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(p.status, WA_STATUS_LAYOUT);
        return;
    }
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);   // [0] tmem base, [1..4] lo min, [5..8] hi max
    float* xbuf = reinterpret_cast<float*>(smem + C::OFF_X);            // [2][2][128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA -> (query tile, head).  Tiles run longest (causal) first; with hfirst the launch order
    // (x fastest, then y) takes every head of a tile before the next, so the longest CTAs of all
    // heads start first instead of the last head's longest ones starting late.
    int bx = static_cast<int>(blockIdx.x), by = static_cast<int>(blockIdx.y);
    if (p.hfirst) {
        const int lin = bx + by * static_cast<int>(gridDim.x);
        bx = lin / static_cast<int>(gridDim.y);
        by = lin % static_cast<int>(gridDim.y);
    }
    const int qt = p.nqt - 1 - bx;
    const int G = p.hq / p.hkv;
    // Dense: one query head, 128 rows, lane = row.  Block-sparse: the key head's G query heads
    // for R = 128 / G rows, lane m = (row m / G, head m % G).
    const int gsz = SP ? p.gsz : 1;
    const int nrows = kBM / gsz;
    const int g = SP ? by : by / G;
    const int h0 = SP ? g * G : by;
    const int m0 = qt * nrows;
    uint32_t* bmap = reinterpret_cast<uint32_t*>(smem + C::OFF_BMAP);
    uint16_t* sel_lists = reinterpret_cast<uint16_t*>(smem + C::OFF_SEL);
    int* sel_cnt = reinterpret_cast<int*>(smem + C::OFF_CNT);
    // block-sparse: the CTA's key span in blocks starts at the first row's window start
    const int j0s = (p.win > 0 ? max(0, p.p0 + m0 - p.win + 1) : 0) / T;
    const int nwords = SP ? (((p.p0 + p.n - 1) / T - j0s) >> 5) + 1 : 1;
    if constexpr (SP) {
        for (int w = threadIdx.x; w < nwords; w += kThreads) bmap[w] = 0u;
    }

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_Q), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(B_KFULL + s), 1);
            mbar_init(BAR(B_VFULL + s), 1);
            mbar_init(BAR(B_VREADY + s), 1);
            mbar_init(BAR(B_SFULL + s), 1);
            mbar_init(BAR(B_SFREE + s), 8);
            mbar_init(BAR(B_XCHG + s), 8);      // one arrival per softmax warp
        }
        mbar_init(BAR(B_PFULL + 0), 8);
        mbar_init(BAR(B_PFULL + 1), 8);
        mbar_init(BAR(B_PVDONE + 0), 1);
        mbar_init(BAR(B_PVDONE + 1), 1);
        mbar_init(BAR(B_DRAIN), 1);
        mbar_init(BAR(B_EPI_L), 8);
        mbar_init(BAR(B_EPI_B), 8);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), C::TMEM_COLS);
        tmem_relinquish();
    }

    // Row ranges (softmax warps; both halves of a row compute the same): row i sees [lo_i, hi_i].
    int row_lo = 1, row_hi = 0;
    const int r = (warp & 3) * 32 + lane;         // the tensor-memory lane of a softmax thread
    const int rl = r / gsz;                       // its row within the CTA
    const int i = m0 + rl;                        // its row
    const int h = h0 + (r - rl * gsz);            // its query head
    const bool lane_ok = i < p.n && rl < nrows;
    if (warp >= 4) {
        if (lane_ok) {
            const int P = p.p0 + i;
            row_lo = p.win > 0 ? max(0, P - p.win + 1) : 0;
            int hv = P;
            if (p.hi) {
                hv = p.hi[i];
                if (hv < P || hv > p.p0 + p.n - 1) {
                    if (warp < 8) atomicOr(p.status, WA_STATUS_BAD_HI);
                    hv = min(max(hv, P), p.p0 + p.n - 1);
                }
            }
            row_hi = hv;
        }
        if (warp < 8) {
            int mn = lane_ok ? row_lo : INT_MAX, mx = lane_ok ? row_hi : INT_MIN;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
                mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
            }
            if (lane == 0) {
                misc[1 + warp - 4] = static_cast<uint32_t>(mn);
                misc[5 + warp - 4] = static_cast<uint32_t>(mx);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = misc[0];
    if (warp == 0 && lane == 0) {   // Q first: it needs nothing the rest of the set-up computes
        prefetch_tensormap(&p.tq);
        prefetch_tensormap(&p.tk);
        prefetch_tensormap(&p.tv);
        mbar_arrive_expect_tx(BAR(B_Q), C::KB * gsz * nrows * 128);   // the box: 64 dims x gsz x nrows
        for (int b = 0; b < C::KB; ++b)
            tma_load_3d(sbase + C::OFF_Q + b * C::Q_BLOCK, &p.tq, b * 64, h0, m0, BAR(B_Q), policy_evict_first());
    }
    int ulo = INT_MAX, uhi = INT_MIN;
    for (int w = 0; w < 4; ++w) {
        ulo = min(ulo, static_cast<int>(misc[1 + w]));
        uhi = max(uhi, static_cast<int>(misc[5 + w]));
    }
    // Key tiles j0..j1 (absolute positions [jT, jT + T)) cover every row's range.
    const int j0 = ulo / T, j1 = uhi / T;
    int ntiles = j1 - j0 + 1;   // >= 1: the first row of a tile always exists (m0 < n)
    // block-sparse: each row's selected blocks with a visible key, sorted and without repeats,
    // relative to j0 (= j0s: the first row has the smallest window start), and their union
    const uint16_t* my_list = sel_lists + rl * kSelMax;
    if constexpr (SP) {
        if (warp >= 4 && warp < 8 && lane_ok && h == h0) {
            const int32_t* srow = p.sel + (static_cast<int64_t>(i) * p.hkv + g) * p.nsel;
            const int cnt = p.nsel <= kSelMax / 2
                                ? build_block_list<kSelMax / 2>(srow, p.nsel, row_lo / T, row_hi / T, j0s,
                                                                sel_lists + rl * kSelMax, bmap)
                                : build_block_list<kSelMax>(srow, p.nsel, row_lo / T, row_hi / T, j0s,
                                                            sel_lists + rl * kSelMax, bmap);
            sel_cnt[rl] = cnt;
        }
        __syncthreads();
        ntiles = 0;
        for (int w = 0; w < nwords; ++w) ntiles += __popc(bmap[w]);
    }

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        const uint64_t pol_kv = policy_evict_last();
        bool ok = true;
        int issued = 0;
        TileWalk<SP> tiles;
        tiles.init(bmap, nwords);
        for (int idx = 0; idx < ntiles && ok; ++idx) {
            const int s = idx & 1, u = idx >> 1;
            const int key0 = (j0 + tiles.next()) * T;
            const int slot0 = p.win > 0 ? key0 % p.ring : key0;
            const bool wrapped = p.win > 0 && slot0 + T > p.ring;
            for (int kv = 0; kv < 2 && ok; ++kv) {
                const uint32_t full = BAR((kv ? B_VFULL : B_KFULL) + s);
                const uint32_t dst = sbase + (kv ? C::OFF_V : C::OFF_K) + s * C::KV_BYTES;
                // a stage is free once the product that read it is done: S of tile idx - 2 for K,
                // P.V of tile idx - 2 for V (their commits are the only ones the MMA warp issues)
                if (u > 0 && !warp_wait(BAR((kv ? B_PVDONE : B_SFULL) + s), (u - 1) & 1, p.status)) {
                    ok = false;
                    break;
                }
                if (!wrapped) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full, C::KV_BYTES);
                        for (int b = 0; b < C::KB; ++b)
                            tma_load_3d(dst + b * C::KV_BLOCK, kv ? &p.tv : &p.tk, b * 64, g, slot0, full, pol_kv);
                    }
                } else {
                    copy_tile_wrapped<D, T>(dst, kv ? p.v : p.k, kv ? p.v_tok : p.k_tok, g, key0, p.ring, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full);
                }
                __syncwarp();
            }
            issued = idx + 1;
        }
        if (lane == 0) {
            // let every TMA copy already issued land before the CTA can exit, whichever role stopped
            // early (after a normal run every one was consumed, and the waits return at once)
            mbar_wait(BAR(B_Q), 0, p.status);
            for (int idx = max(0, issued - 2); idx < issued; ++idx) {
                mbar_wait(BAR(B_KFULL + (idx & 1)), (idx >> 1) & 1, p.status);
                mbar_wait(BAR(B_VFULL + (idx & 1)), (idx >> 1) & 1, p.status);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (one thread)
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(kBM, T, 0, 0, p.neg ? 1u : 0u);
            constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
            bool ok = mbar_wait(BAR(B_Q), 0, p.status);
            for (int idx = 0; ok && idx <= ntiles; ++idx) {
                if (idx < ntiles) {
                    const int s = idx & 1, u = idx >> 1;
                    ok = mbar_wait(BAR(B_KFULL + s), u & 1, p.status);
                    if (ok && idx >= 2) ok = mbar_wait(BAR(B_SFREE + s), (u - 1) & 1, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    // descriptors built once; step kk moves the start address (16-byte units) by a constant
                    const uint64_t a0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
                    const uint64_t b0 = sdesc_sw128(sbase + C::OFF_K + s * C::KV_BYTES, 16, 1024);
                    const uint32_t d_s = tbase + C::S_COL + s * T;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_bf16_ss(d_s, a0 + (((kk >> 2) * C::Q_BLOCK + (kk & 3) * 32) >> 4),
                                    b0 + (((kk >> 2) * C::KV_BLOCK + (kk & 3) * 32) >> 4), idS, kk > 0 ? 1u : 0u);
                    mma_commit(BAR(B_SFULL + s));
                }
                if (idx >= 1) {
                    const int pidx = idx - 1, ps = pidx & 1, pu = pidx >> 1;
                    ok = mbar_wait(BAR(B_PFULL + (pidx & 1)), (pidx >> 1) & 1, p.status);
                    if (ok) ok = mbar_wait(BAR(B_VREADY + ps), pu & 1, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t v0 = sdesc_sw128(sbase + C::OFF_V + ps * C::KV_BYTES, C::KV_BLOCK, 1024);
#pragma unroll
                    for (int half = 0; half < NP; ++half) {
                        const uint32_t pt = tbase + C::p_col(NP > 1 ? half : (pidx & 1));
#pragma unroll
                        for (int kk = 0; kk < T / 16; ++kk)
                            mma_bf16_ts(tbase + C::O_COL, pt + kk * 8, v0 + ((kk * 16 * 128) >> 4), idO,
                                        (pidx > 0 || kk > 0 || half > 0) ? 1u : 0u);
                    }
                    mma_commit(BAR(B_PVDONE + (pidx & 1)));
                }
            }
            // every MMA issued so far has finished before tensor memory can be released
            mma_commit(BAR(B_DRAIN));
            mbar_wait(BAR(B_DRAIN), 0, p.status);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ V rows outside the key union -> 0
        TileWalk<SP> tiles;
        tiles.init(bmap, nwords);
        for (int idx = 0; idx < ntiles; ++idx) {
            const int s = idx & 1, u = idx >> 1;
            if (!warp_wait(BAR(B_VFULL + s), u & 1, p.status)) break;
            const int key0 = (j0 + tiles.next()) * T;
            const int z_lo = min(T, max(0, ulo - key0));              // rows [0, z_lo)
            const int z_hi = max(0, min(T, uhi - key0 + 1));          // rows [z_hi, T)
            if (z_lo > 0 || z_hi < T) {
                const uint32_t vst = sbase + C::OFF_V + s * C::KV_BYTES;
                const int nz = z_lo + (T - z_hi);
                for (int u16 = lane; u16 < nz * C::KB * 8; u16 += 32) {
                    const int zr = u16 / (C::KB * 8);
                    const int rem = u16 % (C::KB * 8);
                    const int row = zr < z_lo ? zr : z_hi + (zr - z_lo);
                    st_shared_v4(vst + (rem / 8) * C::KV_BLOCK + row * 128 + (rem % 8) * 16, 0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_VREADY + s));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ softmax: row r, column half wg
        const int wg = (warp - 4) >> 2;
        const int col0 = wg * NC;                                    // first S column of this half
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float c = p.c;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        TileWalk<SP> tiles;
        tiles.init(bmap, nwords);
        int sel_ptr = 0;
        const int sel_n = (SP && lane_ok) ? sel_cnt[rl] : 0;
        for (int idx = 0; ok && idx < ntiles; ++idx) {
            const int s = idx & 1, u = idx >> 1;
            if (!warp_wait(BAR(B_SFULL + s), u & 1, p.status)) { ok = false; break; }
            tc_fence_after();
            float sv[NC];
            load_s<NC>(tbase + lane_addr + C::S_COL + s * T + col0, sv);

            // visible columns of this half: [vlo, vhi]; interior tiles need no mask at all
            const int rel = tiles.next();
            const int kbase = (j0 + rel) * T + col0;
            int vlo = row_lo - kbase, vhi = row_hi - kbase;
            if constexpr (SP) {   // a block the row did not select is masked whole
                if (sel_ptr < sel_n && my_list[sel_ptr] == rel) {
                    ++sel_ptr;
                } else {
                    vlo = NC;
                    vhi = -1;
                }
            }
            const bool masked = !__all_sync(0xFFFFFFFFu, vlo <= 0 && vhi >= NC - 1);
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
            if (masked) {
#pragma unroll
                for (int k = 0; k < NC; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], (k >= vlo && k <= vhi) ? sv[k] : -INFINITY);
            } else {
#pragma unroll
                for (int k = 0; k < NC; k += 2) mx8[(k >> 1) & 7] = max3(mx8[(k >> 1) & 7], sv[k], sv[k + 1]);
            }
            const float mh = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            // exchange the half-row maxima (raw S units) with the other half
            float* xs = xbuf + (idx & 1) * (2 * kBM);
            xs[wg * kBM + r] = mh;
            __syncwarp();   // the warp's stores precede lane 0's (cumulative) release
            if (lane == 0) mbar_arrive(BAR(B_XCHG + (idx & 1)));
            float ls8[8];
            // p = 2^(S c - m_sub) into sv, and the row sum in ls8
            auto exponents = [&](float m_sub) {
#pragma unroll
                for (int e = 0; e < 8; ++e) ls8[e] = 0.f;
                if (masked) {   // a masked column is 0 whatever its score (also for scale 0 or a NaN key)
#pragma unroll
                    for (int k = 0; k < NC; ++k) {
                        const float pk = (k >= vlo && k <= vhi) ? ex2(fmaf(sv[k], c, -m_sub)) : 0.f;
                        sv[k] = pk;
                        ls8[k & 7] += pk;
                    }
                } else {   // two columns per packed FMA and packed add
#pragma unroll
                    for (int k = 0; k < NC; k += 2) {
                        float x0, x1;
                        fma_x2(x0, x1, sv[k], sv[k + 1], c, c, -m_sub, -m_sub);
                        sv[k] = ex2(x0);
                        sv[k + 1] = ex2(x1);
                        const int j = (k >> 1) & 3;
                        add_x2(ls8[2 * j], ls8[2 * j + 1], sv[k], sv[k + 1]);
                    }
                }
            };
            // The lazy rule usually keeps the running max, so the exponentials start with it while
            // the other half's maximum is on its way; a warp in which any row's max moves redoes
            // them from the S buffer (still held: SFREE comes after).  The values are those of the
            // rule's own m either way.
            const bool spec = __all_sync(0xFFFFFFFFu, m_run != -INFINITY && mh * c <= m_run + kLazy);
            if (spec) exponents(m_run);
            if (!warp_wait(BAR(B_XCHG + (idx & 1)), (idx >> 1) & 1, p.status)) { ok = false; break; }
            const float mraw = fmaxf(xs[r], xs[kBM + r]);   // the same order in both halves
            const float mt = mraw * c;                       // tile max in log2 units
            // lazy rescale: keep the running max unless the tile's exceeds it by more than kLazy
            const float m_new = (mt > m_run + kLazy) ? mt : m_run;
            const float alpha = (m_new == m_run) ? 1.f : ex2(m_run - m_new);
            const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
            if (!spec || __any_sync(0xFFFFFFFFu, m_new != m_run)) {
                if (spec) load_s<NC>(tbase + lane_addr + C::S_COL + s * T + col0, sv);
                exponents(m_sub);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_SFREE + s));
            const float lsum = ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
            l_run = (alpha == 1.f) ? (l_run + lsum) : fmaf(l_run, alpha, lsum);
            m_run = m_new;

            // P buffer reuse: the P.V that last read it (tile idx - P_BUFS) must be done
            const int reuse = idx - C::P_BUFS;
            if (reuse >= 0) {
                if (!warp_wait(BAR(B_PVDONE + (reuse & 1)), (reuse >> 1) & 1, p.status)) { ok = false; break; }
                tc_fence_after();
            }
            // an O rescale must wait for the previous tile's P.V (already covered when P_BUFS is 1)
            if (idx >= 1 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
                if (C::P_BUFS == 2) {
                    if (!warp_wait(BAR(B_PVDONE + ((idx - 1) & 1)), ((idx - 1) >> 1) & 1, p.status)) { ok = false; break; }
                    tc_fence_after();
                }
                {
#pragma unroll 1
                    for (int cc = 0; cc < D / 64; ++cc) {
                        uint32_t o[32];
                        const uint32_t ta = tbase + lane_addr + C::O_COL + wg * (D / 2) + cc * 32;
                        tmem_ld32_wait(ta, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(ta, o);
                    }
                    tmem_wait_st();
                }
            }
            // P (and its residual parts) into tensor memory, two bf16 per column, this thread's
            // columns.  Each residual p - part is exact in fp32.
            {
                uint32_t w[NP][NC / 2];
#pragma unroll
                for (int e = 0; e < NC / 2; ++e) {
                    float a = sv[2 * e], b = sv[2 * e + 1];
#pragma unroll
                    for (int part = 0; part < NP; ++part) {
                        w[part][e] = pack_bf16(a, b);
                        a -= __uint_as_float(w[part][e] << 16);
                        b -= __uint_as_float(w[part][e] & 0xFFFF0000u);
                    }
                }
#pragma unroll
                for (int part = 0; part < NP; ++part) {
                    const uint32_t pa = tbase + lane_addr + C::p_col(NP > 1 ? part : (idx & 1)) + col0 / 2;
                    if constexpr (NC == 64) tmem_st32(pa, w[part]);
                    else tmem_st16(pa, w[part]);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_PFULL + (idx & 1)));
        }
        // epilogue: l = l(half 0) + l(half 1); o = O / l, bf16; a non-finite row goes to the float64 re-run
        if (SP && ntiles == 0) {
            // block-sparse, no selected key visible to any row of the CTA: every output is 0 / 0
            if (lane_ok) {
                uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(i) * p.o_tok +
                                                      static_cast<int64_t>(h) * D + wg * (D / 2));
                for (int e = 0; e < D / 16; ++e) dst[e] = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
                if (wg == 0) p.flags[atomicAdd(p.nflag, 1)] = i * p.hq + h;
            }
            ok = false;
        }
        if (ok) ok = warp_wait(BAR(B_PVDONE + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, p.status);
        float* xl = xbuf + ((ntiles & 1) ^ 0) * (2 * kBM);   // the buffer the last tile did not use
        if (ok) {
            xl[wg * kBM + r] = l_run;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_EPI_L));
            ok = warp_wait(BAR(B_EPI_L), 0, p.status);
        }
        if (ok) {
            const float l = xl[r] + xl[kBM + r];
            // o = O / l as O times the correctly rounded 1 / l: within one fp32 ulp of the quotient,
            // far inside the bf16 rounding that follows, for one division a row instead of d / 2
            const float inv_l = __fdiv_rn(1.f, l);
            tc_fence_after();
            bool bad = false;
            uint16_t* orow = p.out + static_cast<int64_t>(i) * p.o_tok + static_cast<int64_t>(h) * D + wg * (D / 2);
#pragma unroll 1
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t o[32];
                tmem_ld32_wait(tbase + lane_addr + C::O_COL + wg * (D / 2) + cc * 32, o);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float a = __uint_as_float(o[2 * e]) * inv_l;
                    const float b = __uint_as_float(o[2 * e + 1]) * inv_l;
                    bad |= !(isfinite(a) && isfinite(b));
                    pk[e] = pack_bf16(a, b);
                }
                if (lane_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            // both halves' verdicts meet in the other exchange buffer; half 0 queues the row
            int* xb = reinterpret_cast<int*>(xbuf + ((ntiles & 1) ^ 1) * (2 * kBM));
            xb[wg * kBM + r] = bad ? 1 : 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_EPI_B));
            if (warp_wait(BAR(B_EPI_B), 0, p.status) && wg == 0 && lane_ok && (xb[r] | xb[kBM + r])) {
                const int slot = atomicAdd(p.nflag, 1);
                p.flags[slot] = i * p.hq + h;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, C::TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
    g_encode = tensor_map_encoder();
    return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// A [tokens, heads, d] bf16 view with token stride `tok` elements; box of 64 x box_heads x rows.
bool encode_3d(CUtensorMap* m, const void* base, int d, int heads, int tokens, int64_t tok, int rows,
               int box_heads = 1) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(tok) * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(rows)};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int NP, bool SP>
cudaError_t launch_t(const PromptArgs& a, cudaStream_t s) {
    using C = Cfg<D, NP, SP>;
    PromptParams pp{};
    // block-sparse: the G query heads of a key head share the CTA, for 128 / G rows
    const int gsz = SP ? a.hq / a.hkv : 1;
    const int rows = kBM / gsz;
    if (!encode_3d(&pp.tq, a.q, D, a.hq, a.n, a.q_tok, rows, gsz) ||
        !encode_3d(&pp.tk, a.k, D, a.hkv, a.ring, a.k_tok, C::T) ||
        !encode_3d(&pp.tv, a.v, D, a.hkv, a.ring, a.v_tok, C::T))
        return cudaErrorInvalidValue;
    pp.k = static_cast<const uint16_t*>(a.k);
    pp.v = static_cast<const uint16_t*>(a.v);
    pp.hi = a.hi;
    pp.out = static_cast<uint16_t*>(a.out);
    pp.status = &a.hdr->status;
    pp.nflag = &a.hdr->nflag;
    pp.flags = a.flags;
    pp.k_tok = a.k_tok;
    pp.v_tok = a.v_tok;
    pp.o_tok = a.o_tok;
    pp.p0 = a.p0; pp.n = a.n; pp.hq = a.hq; pp.hkv = a.hkv; pp.win = a.win; pp.ring = a.ring;
    pp.nqt = (a.n + rows - 1) / rows;
    pp.neg = a.scale < 0.f ? 1 : 0;
    pp.c = (a.scale < 0.f ? -a.scale : a.scale) * 1.4426950408889634f;
    pp.sel = a.sel;
    pp.nsel = a.nsel;
    pp.gsz = gsz;
    // causal on a linear cache: CTA lengths grow with the tile, so all heads' longest go first
    pp.hfirst = (!SP && a.win == 0 && a.hi == nullptr) ? 1 : 0;
    const dim3 grid(pp.nqt, SP ? a.hkv : a.hq);
    prompt_kernel<D, NP, SP><<<grid, kThreads, C::SMEM, s>>>(pp);
    return cudaGetLastError();
}

template <int D, int NP, bool SP = false>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(prompt_kernel<D, NP, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<D, NP, SP>::SMEM);
}

}  // namespace

}  // namespace wa
