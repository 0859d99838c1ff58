// wa_prompt_d256.cuh — the prompt kernel at head dim 256 with one or two P parts: 128-key tiles,
// P written over S, K and V staged through a ring of half-tile slots in the order the tensor core
// reads them.
//
// What it computes is the prompt form of wa_prompt_kernel.cuh (TensorFold pull request #1123,
// "What this changes": bullets "Prompt", "Window.p32", "promptRows(..., hi)", "Scale is a
// parameter"): key tiles at absolute positions, each folded into a row's running softmax once,
// fp32 probabilities, P entering P.V as bf16(P) or bf16(P) + bf16(P - bf16(P)).  A row's fp32
// sums run over the same absolute 128-key tiles in key order whoever shares its CTA, so its bits
// do not depend on the batch or on where a prompt is cut.
//
// GB300 layout (one CTA per 128-row query tile of one query head, 384 threads):
//   tensor memory   O [0, 256)   S0 [256, 384)   S1 [384, 512)   (fp32 columns)
//                   S of key tile j goes to buffer j & 1; P of tile j is written over it: keys
//                   [64 h, 64 h + 64) of part k at column 64 h + 32 k, two bf16 per column.
//   shared memory   Q (64 KiB: four 64-dim blocks of 128 rows), then a ring of five 32 KiB slots.
//                   A slot holds half an operand: K rows of 128 keys x 128 dims (two 64-dim
//                   blocks) or V rows of 64 keys x 256 dims (four blocks), 128-byte swizzle.
//                   Halves are loaded in the order the tensor core consumes them:
//                   K0, K1, V0, K2, V1, K3, V2, ..., so every slot is released in load order
//                   and each load is issued about one and a half tiles before it is needed.
//   warp 0          TMA producer: Q once, then the half-operands into the ring; halves that wrap
//                   around the ring's end are copied by the warp with the same swizzle.
//   warp 1          allocates tensor memory; lane 0 issues, per key tile j,
//                     S(j + 1) = Q K(j + 1)^T   (N = 128: sixteen K steps)
//                     O += P(j) V(j)            (N = 256, in two 64-key halves, every P part)
//                   so the softmax of tile j runs while S(j + 1) and the previous P.V execute.
//                   A commit after each half-operand's products releases its slot.
//   warp 2          zeroes V rows outside the CTA's key union (first and last tile).
//   warps 4..11     two warpgroups, one per 64-column half of the tile: warp w owns tensor-memory
//                   lanes 32 (w % 4) .. + 31 (rows), warpgroup g columns [64 g, 64 g + 64).  The
//                   half-row maxima meet in shared memory; then exponentials, P over the half's
//                   own S columns, the lazy O rescale of the half's own O columns, epilogue.
// Every wait is bounded (a status bit after kWaitLimitNs) and warp-uniform where a warp waits.
#pragma once

#include "wa_prompt_kernel.cuh"

namespace wa {

namespace {

template <int NP>
struct WideCfg {
    static constexpr int D = 256, T = 128;
    static constexpr int Q_BLOCK = kBM * 128;                   // one 64-dim block of Q: 16 KiB
    static constexpr int Q_BYTES = 4 * Q_BLOCK;
    static constexpr int NSLOT = 5;
    static constexpr int SLOT = 32768;
    static constexpr int K_BLOCK = T * 128;                     // K half: [2 blocks][128 keys][128 B]
    static constexpr int V_BLOCK = (T / 2) * 128;               // V half: [4 blocks][64 keys][128 B]
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = OFF_Q + Q_BYTES;
    static constexpr int OFF_X = OFF_RING + NSLOT * SLOT;       // row exchange [2 tiles][2 halves][128] fp32
    static constexpr int OFF_BAR = OFF_X + 2 * 2 * kBM * 4;
    static constexpr int NBAR = 32;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;         // tmem base, per-warp union bounds
    static constexpr int SMEM = OFF_MISC + 64;
    static constexpr int TMEM_COLS = 512;
    static constexpr int O_COL = 0;
    __host__ __device__ static constexpr int s_col(int b) { return D + b * T; }
    static_assert(NP == 1 || NP == 2, "P parts over S: 32 columns per 64 keys each");
    static_assert(s_col(1) + T <= TMEM_COLS, "tensor memory budget");
    static_assert(2 * K_BLOCK == SLOT && 4 * V_BLOCK == SLOT, "half-operands fill a slot");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// Barrier indices.  FREE per ring slot (the producer takes every use of a slot in order); [b] = per
// key-tile parity (tile & 1); KFULL, VFULL and VREADY per operand half and tile parity.  A parity
// wait for phase k is only sound while the barrier has completed phase k - 1 and cannot have
// completed phase k + 1.  A slot holds K and V halves in turn, so a per-slot "loaded" barrier would
// let the V sanitizer (which waits for V halves only) meet a slot whose previous, K, load had not
// landed yet and take that phase for its own; loads therefore signal per operand half and tile
// parity, whose phases each waiter takes in order.
enum : int {
    WB_Q = 0, WB_KFULL = 1, WB_VFULL = 5, WB_FREE = 9, WB_SFULL = 14, WB_PVDONE = 16,   // K/VFULL [half][b]
    WB_VREADY = 18,  // [half][b]
    WB_XCHG = 22, WB_PHALF = 24, WB_PFULL = 26, WB_EPI_L = 28, WB_EPI_B = 29, WB_DRAIN = 30
};

// The ring's load sequence is K0, then for each tile j: K(j + 1) if it exists, then V(j).
// Operand index of K(j) and of V(j) in that sequence (two half-loads each).
__device__ __forceinline__ int op_of_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int op_of_v(int j, int ntiles) { return j + 1 < ntiles ? 2 * j + 2 : 2 * j + 1; }

// Copy nkeys key rows (slots (key0 + k) mod ring) of dims [dim0, dim0 + 64 nblocks) into a swizzled
// slot laid out [block][key][128 B], by one warp.  Used where a half-operand wraps around the end
// of the ring, which one TMA box cannot express.
__device__ void copy_half_wrapped(uint32_t dst, const uint16_t* base, int64_t tok, int g, int key0, int nkeys,
                                  int dim0, int nblocks, int ring, int lane) {
    const int units = nkeys * nblocks * 8;   // 16-byte units
    for (int u = lane; u < units; u += 32) {
        const int k = u / (nblocks * 8);
        const int rem = u % (nblocks * 8);
        const int b = rem / 8, c = rem % 8;
        const int slot = (key0 + k) % ring;
        const uint4 val = ld_global_nc_v4(base + slot * tok + static_cast<int64_t>(g) * 256 + dim0 + b * 64 + c * 8);
        st_shared_v4(dst + b * (nkeys * 128) + k * 128 + ((c ^ (k & 7)) * 16), val.x, val.y, val.z, val.w);
    }
    fence_proxy_async_smem();
}

template <int NP>
__global__ void __launch_bounds__(kThreads, 1) prompt_d256_kernel(const __grid_constant__ PromptParams p) {
    using C = WideCfg<NP>;
    constexpr int D = C::D, T = C::T;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {   // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(p.status, WA_STATUS_LAYOUT);
        return;
    }
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    auto SLOT = [&](int s) { return sbase + C::OFF_RING + static_cast<uint32_t>(s) * C::SLOT; };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);   // [0] tmem base, [1..4] lo min, [5..8] hi max
    float* xbuf = reinterpret_cast<float*>(smem + C::OFF_X);            // [2][2][128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA -> (query tile, head): longest (causal) tiles first; with hfirst every head of a tile
    // goes before the next tile, so the longest CTAs of all heads start first.
    int bx = static_cast<int>(blockIdx.x), by = static_cast<int>(blockIdx.y);
    if (p.hfirst) {
        const int lin = bx + by * static_cast<int>(gridDim.x);
        bx = lin / static_cast<int>(gridDim.y);
        by = lin % static_cast<int>(gridDim.y);
    }
    const int qt = p.nqt - 1 - bx;
    const int h = by;
    const int g = h / (p.hq / p.hkv);
    const int m0 = qt * kBM;

    if (threadIdx.x == 0) {
        mbar_init(BAR(WB_Q), 1);
        for (int s = 0; s < C::NSLOT; ++s) mbar_init(BAR(WB_FREE + s), 1);
        for (int x = 0; x < 4; ++x) {
            mbar_init(BAR(WB_KFULL + x), 1);      // [half][b]: TMA bytes, or one arrival after a warp copy
            mbar_init(BAR(WB_VFULL + x), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(BAR(WB_SFULL + b), 1);      // MMA commits
            mbar_init(BAR(WB_PVDONE + b), 1);
            mbar_init(BAR(WB_VREADY + b), 1);     // [half 0][b]
            mbar_init(BAR(WB_VREADY + 2 + b), 1); // [half 1][b]
            mbar_init(BAR(WB_XCHG + b), 8);       // one arrival per softmax warp
            mbar_init(BAR(WB_PHALF + b), 8);      // keys 0..63 of P and all of O's rescale in place
            mbar_init(BAR(WB_PFULL + b), 4);      // keys 64..127 of P in place
        }
        mbar_init(BAR(WB_EPI_L), 8);
        mbar_init(BAR(WB_EPI_B), 8);
        mbar_init(BAR(WB_DRAIN), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), C::TMEM_COLS);
        tmem_relinquish();
    }

    // softmax threads: row r of the tile (= tensor-memory lane), columns of half wg
    const int r = (warp & 3) * 32 + lane;
    const int i = m0 + r;
    const bool lane_ok = i < p.n;
    int row_lo = 1, row_hi = 0;
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
        mbar_arrive_expect_tx(BAR(WB_Q), C::Q_BYTES);
        for (int b = 0; b < 4; ++b)
            tma_load_3d(sbase + C::OFF_Q + b * C::Q_BLOCK, &p.tq, b * 64, h, m0, BAR(WB_Q), policy_evict_first());
    }
    int ulo = INT_MAX, uhi = INT_MIN;
    for (int w = 0; w < 4; ++w) {
        ulo = min(ulo, static_cast<int>(misc[1 + w]));
        uhi = max(uhi, static_cast<int>(misc[5 + w]));
    }
    // Key tiles j0..j1 (absolute positions [jT, jT + T)) cover every row's range.
    const int j0 = ulo / T;
    const int ntiles = uhi / T - j0 + 1;   // >= 1: the CTA's first row exists (m0 < n)
    const int nhalf = 4 * ntiles;          // half-loads in the ring sequence

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        const uint64_t pol_kv = policy_evict_last();
        bool ok = true;
        int issued = 0;
        int lastbar[C::NSLOT], lastph[C::NSLOT];   // the barrier and phase of the load in each slot
        for (int u = 0; u < nhalf && ok; ++u) {
            const int o = u >> 1, half = u & 1;
            // operand o of the sequence K0, K1, V0, K2, V1, ...: K(t) or V(t)
            bool is_v;
            int t;
            if (o == 0) {
                is_v = false;
                t = 0;
            } else if (o == 2 * ntiles - 1) {
                is_v = true;
                t = ntiles - 1;
            } else {
                is_v = (o & 1) == 0;
                t = is_v ? (o - 2) >> 1 : (o + 1) >> 1;
            }
            const int s = u % C::NSLOT, use = u / C::NSLOT;
            if (use > 0 && !warp_wait(BAR(WB_FREE + s), (use - 1) & 1, p.status)) {
                ok = false;
                break;
            }
            // loaded: signalled per operand half and tile parity
            const int fb = (is_v ? WB_VFULL : WB_KFULL) + 2 * half + (t & 1);
            lastbar[s] = fb;
            lastph[s] = (t >> 1) & 1;
            const uint32_t full = BAR(fb);
            const uint32_t dst = SLOT(s);
            const int key0 = (j0 + t) * T + (is_v ? half * 64 : 0);
            const int nkeys = is_v ? 64 : T;
            const int slot0 = p.win > 0 ? key0 % p.ring : key0;
            const bool wrapped = p.win > 0 && slot0 + nkeys > p.ring;
            if (!wrapped) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(full, C::SLOT);
                    if (is_v) {
                        for (int b = 0; b < 4; ++b)
                            tma_load_3d(dst + b * C::V_BLOCK, &p.tv, b * 64, g, slot0, full, pol_kv);
                    } else {
                        for (int b = 0; b < 2; ++b)
                            tma_load_3d(dst + b * C::K_BLOCK, &p.tk, half * 128 + b * 64, g, slot0, full, pol_kv);
                    }
                }
            } else {
                if (is_v)
                    copy_half_wrapped(dst, p.v, p.v_tok, g, key0, 64, 0, 4, p.ring, lane);
                else
                    copy_half_wrapped(dst, p.k, p.k_tok, g, key0, T, half * 128, 2, p.ring, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(full);
            }
            __syncwarp();
            issued = u + 1;
        }
        if (lane == 0) {
            // let every copy already issued land before the CTA can exit, whichever role stopped
            // early (after a normal run every one was consumed, and the waits return at once): the
            // last NSLOT loads hold one slot each
            mbar_wait(BAR(WB_Q), 0, p.status);
            for (int u = max(0, issued - C::NSLOT); u < issued; ++u)
                mbar_wait(BAR(lastbar[u % C::NSLOT]), lastph[u % C::NSLOT], p.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (one thread)
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(kBM, T, 0, 0, p.neg ? 1u : 0u);
            constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
            const uint64_t aq = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
            // S(t) = Q K(t)^T into buffer t & 1: K steps 0..7 read the first K half, 8..15 the second;
            // each half's products are followed by a commit that frees its slot.
            auto issue_s = [&](int t) -> bool {
                const uint32_t d_s = tbase + C::s_col(t & 1);
#pragma unroll
                for (int kh = 0; kh < 2; ++kh) {
                    const int u = 2 * op_of_k(t) + kh, s = u % C::NSLOT;
                    if (!mbar_wait(BAR(WB_KFULL + 2 * kh + (t & 1)), (t >> 1) & 1, p.status)) return false;
                    tc_fence_after();
                    const uint64_t bk = sdesc_sw128(SLOT(s), 16, 1024);
#pragma unroll
                    for (int k8 = 0; k8 < 8; ++k8) {
                        const int kk = 8 * kh + k8;
                        mma_bf16_ss(d_s, aq + (((kk >> 2) * C::Q_BLOCK + (kk & 3) * 32) >> 4),
                                    bk + ((((k8 >> 2) & 1) * C::K_BLOCK + (k8 & 3) * 32) >> 4), idS,
                                    kk > 0 ? 1u : 0u);
                    }
                    mma_commit(BAR(WB_FREE + s));
                }
                mma_commit(BAR(WB_SFULL + (t & 1)));
                return true;
            };
            // O += P(t) V(t) over one 64-key half hh (K steps 4 hh .. 4 hh + 3 of every P part).
            auto issue_pv_half = [&](int t, int hh) -> bool {
                const int b = t & 1;
                if (!mbar_wait(BAR(WB_VREADY + 2 * hh + b), (t >> 1) & 1, p.status)) return false;
                if (!mbar_wait(BAR((hh ? WB_PFULL : WB_PHALF) + b), (t >> 1) & 1, p.status)) return false;
                tc_fence_after();
                const int u = 2 * op_of_v(t, ntiles) + hh, s = u % C::NSLOT;
                const uint64_t v0 = sdesc_sw128(SLOT(s), C::V_BLOCK, 1024);
#pragma unroll
                for (int part = 0; part < NP; ++part)
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        mma_bf16_ts(tbase + C::O_COL, tbase + C::s_col(b) + hh * 64 + part * 32 + k4 * 8,
                                    v0 + ((k4 * 16 * 128) >> 4), idO, (t > 0 || hh > 0 || part > 0 || k4 > 0) ? 1u : 0u);
                mma_commit(BAR(WB_FREE + s));
                if (hh == 1) mma_commit(BAR(WB_PVDONE + b));
                return true;
            };
            bool ok = mbar_wait(BAR(WB_Q), 0, p.status) && issue_s(0);
            for (int t = 0; ok && t < ntiles; ++t) {
                // S(t + 1) overwrites buffer (t + 1) & 1, which held P(t - 1): O += P(t - 1) V(t - 1)
                // was issued before it, and the tensor core runs one thread's products in order.
                if (t + 1 < ntiles) ok = issue_s(t + 1);
                if (ok) ok = issue_pv_half(t, 0);
                if (ok) ok = issue_pv_half(t, 1);
            }
            // every MMA issued so far has finished before tensor memory can be released
            mma_commit(BAR(WB_DRAIN));
            mbar_wait(BAR(WB_DRAIN), 0, p.status);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ V rows outside the key union -> 0
        for (int t = 0; t < ntiles; ++t) {
            bool ok = true;
            for (int hh = 0; hh < 2; ++hh) {
                const int u = 2 * op_of_v(t, ntiles) + hh, s = u % C::NSLOT;
                if (!warp_wait(BAR(WB_VFULL + 2 * hh + (t & 1)), (t >> 1) & 1, p.status)) {
                    ok = false;
                    break;
                }
                const int key0 = (j0 + t) * T + 64 * hh;
                const int z_lo = min(64, max(0, ulo - key0));             // rows [0, z_lo)
                const int z_hi = max(0, min(64, uhi - key0 + 1));         // rows [z_hi, 64)
                if (z_lo > 0 || z_hi < 64) {
                    const uint32_t vst = SLOT(s);
                    const int nz = z_lo + (64 - z_hi);
                    for (int u16 = lane; u16 < nz * 4 * 8; u16 += 32) {
                        const int zr = u16 / (4 * 8);
                        const int rem = u16 % (4 * 8);
                        const int row = zr < z_lo ? zr : z_hi + (zr - z_lo);
                        st_shared_v4(vst + (rem / 8) * C::V_BLOCK + row * 128 + (rem % 8) * 16, 0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(WB_VREADY + 2 * hh + (t & 1)));
            }
            if (!ok) break;
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ softmax: row r, column half wg
        const int wg = (warp - 4) >> 2;
        const int col0 = wg * 64;                                     // first S column (key) of this half
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float c = p.c;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int t = 0; ok && t < ntiles; ++t) {
            const int b = t & 1;
            if (!warp_wait(BAR(WB_SFULL + b), (t >> 1) & 1, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t t_s = tbase + lane_addr + C::s_col(b) + col0;
            float sv[64];
            {
                uint32_t raw[64];
                tmem_ld64_wait(t_s, raw);
#pragma unroll
                for (int e = 0; e < 64; ++e) sv[e] = __uint_as_float(raw[e]);
            }
            // visible columns of this half: [vlo, vhi]; interior tiles need no mask at all
            const int kbase = (j0 + t) * T + col0;
            const int vlo = row_lo - kbase, vhi = row_hi - kbase;
            const bool masked = !__all_sync(0xFFFFFFFFu, vlo <= 0 && vhi >= 63);
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
            if (masked) {
#pragma unroll
                for (int k = 0; k < 64; ++k) mx8[k & 7] = fmaxf(mx8[k & 7], (k >= vlo && k <= vhi) ? sv[k] : -INFINITY);
            } else {
#pragma unroll
                for (int k = 0; k < 64; k += 2) mx8[(k >> 1) & 7] = max3(mx8[(k >> 1) & 7], sv[k], sv[k + 1]);
            }
            const float mh = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            // exchange the half-row maxima (raw S units) with the other half
            float* xs = xbuf + b * (2 * kBM);
            xs[wg * kBM + r] = mh;
            __syncwarp();   // the warp's stores precede lane 0's (cumulative) release
            if (lane == 0) mbar_arrive(BAR(WB_XCHG + b));
            float ls8[8];
            // p = 2^(S c - m_sub) into sv, and the half row's sum in ls8
            auto exponents = [&](float m_sub) {
#pragma unroll
                for (int e = 0; e < 8; ++e) ls8[e] = 0.f;
                if (masked) {   // a masked column is 0 whatever its score (also for scale 0 or a NaN key)
#pragma unroll
                    for (int k = 0; k < 64; ++k) {
                        const float pk = (k >= vlo && k <= vhi) ? ex2(fmaf(sv[k], c, -m_sub)) : 0.f;
                        sv[k] = pk;
                        ls8[k & 7] += pk;
                    }
                } else {   // two columns per packed FMA and packed add
#pragma unroll
                    for (int k = 0; k < 64; k += 2) {
                        float x0, x1;
                        fma_x2(x0, x1, sv[k], sv[k + 1], c, c, -m_sub, -m_sub);
                        sv[k] = ex2(x0);
                        sv[k + 1] = ex2(x1);
                        const int jj = (k >> 1) & 3;
                        add_x2(ls8[2 * jj], ls8[2 * jj + 1], sv[k], sv[k + 1]);
                    }
                }
            };
            // The lazy rule usually keeps the running max, so the exponentials start with it while
            // the other half's maximum is on its way; a warp in which any row's max moves redoes
            // them from S (still in tensor memory: P is written over it only below).
            const bool spec = __all_sync(0xFFFFFFFFu, m_run != -INFINITY && mh * c <= m_run + kLazy);
            if (spec) exponents(m_run);
            if (!warp_wait(BAR(WB_XCHG + b), (t >> 1) & 1, p.status)) { ok = false; break; }
            const float mraw = fmaxf(xs[r], xs[kBM + r]);   // the same order in both halves
            const float mt = mraw * c;                       // tile max in log2 units
            // lazy rescale: keep the running max unless the tile's exceeds it by more than kLazy
            const float m_new = (mt > m_run + kLazy) ? mt : m_run;
            const float alpha = (m_new == m_run) ? 1.f : ex2(m_run - m_new);
            const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
            if (!spec || __any_sync(0xFFFFFFFFu, m_new != m_run)) {
                if (spec) {
                    uint32_t raw[64];
                    tmem_ld64_wait(t_s, raw);
#pragma unroll
                    for (int e = 0; e < 64; ++e) sv[e] = __uint_as_float(raw[e]);
                }
                exponents(m_sub);
            }
            // O rescale of this half's O columns [128 wg, 128 wg + 128), once the previous P.V is done;
            // P.V of this tile waits for it through the half-P barrier (all eight warps arrive there)
            if (t >= 1 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
                if (!warp_wait(BAR(WB_PVDONE + ((t - 1) & 1)), ((t - 1) >> 1) & 1, p.status)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    const uint32_t ta = tbase + lane_addr + C::O_COL + wg * 128 + cc * 32;
                    tmem_ld32_wait(ta, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(ta, o);
                }
                tmem_wait_st();
            }
            if (wg == 1) {   // the second half's O columns are ready for this tile's first P.V half
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(WB_PHALF + b));
            }
            // P over this half's own S columns (already read): part k at column 32 k, two bf16 per
            // column.  The residual p - hi is exact in fp32.
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t w[NP][16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float a = sv[cc * 32 + 2 * e], bb = sv[cc * 32 + 2 * e + 1];
#pragma unroll
                    for (int part = 0; part < NP; ++part) {
                        w[part][e] = pack_bf16(a, bb);
                        a -= __uint_as_float(w[part][e] << 16);
                        bb -= __uint_as_float(w[part][e] & 0xFFFF0000u);
                    }
                }
#pragma unroll
                for (int part = 0; part < NP; ++part) tmem_st16(t_s + part * 32 + cc * 16, w[part]);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR((wg == 0 ? WB_PHALF : WB_PFULL) + b));
            const float lsum = ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
            l_run = (alpha == 1.f) ? (l_run + lsum) : fmaf(l_run, alpha, lsum);
            m_run = m_new;
        }
        // epilogue: l = l(half 0) + l(half 1); o = O / l, bf16; a non-finite row goes to the float64 re-run
        if (ok) ok = warp_wait(BAR(WB_PVDONE + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, p.status);
        float* xl = xbuf + (ntiles & 1) * (2 * kBM);   // the buffer the last tile did not use
        if (ok) {
            xl[wg * kBM + r] = l_run;
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(WB_EPI_L));
            ok = warp_wait(BAR(WB_EPI_L), 0, p.status);
        }
        if (ok) {
            const float l = xl[r] + xl[kBM + r];
            // o = O / l as O times the correctly rounded 1 / l: within one fp32 ulp of the quotient,
            // far inside the bf16 rounding that follows, for one division a row instead of d / 2
            const float inv_l = __fdiv_rn(1.f, l);
            tc_fence_after();
            bool bad = false;
            uint16_t* orow = p.out + static_cast<int64_t>(i) * p.o_tok + static_cast<int64_t>(h) * D + wg * 128;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                tmem_ld32_wait(tbase + lane_addr + C::O_COL + wg * 128 + cc * 32, o);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float a = __uint_as_float(o[2 * e]) * inv_l;
                    const float bb = __uint_as_float(o[2 * e + 1]) * inv_l;
                    bad |= !(isfinite(a) && isfinite(bb));
                    pk[e] = pack_bf16(a, bb);
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
            if (lane == 0) mbar_arrive(BAR(WB_EPI_B));
            if (warp_wait(BAR(WB_EPI_B), 0, p.status) && wg == 0 && lane_ok && (xb[r] | xb[kBM + r])) {
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

template <int NP>
cudaError_t launch_d256(const PromptArgs& a, cudaStream_t s) {
    using C = WideCfg<NP>;
    PromptParams pp{};
    if (!encode_3d(&pp.tq, a.q, C::D, a.hq, a.n, a.q_tok, kBM) ||
        !encode_3d(&pp.tk, a.k, C::D, a.hkv, a.ring, a.k_tok, C::T) ||
        !encode_3d(&pp.tv, a.v, C::D, a.hkv, a.ring, a.v_tok, C::T / 2))
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
    pp.nqt = (a.n + kBM - 1) / kBM;
    pp.neg = a.scale < 0.f ? 1 : 0;
    pp.c = (a.scale < 0.f ? -a.scale : a.scale) * 1.4426950408889634f;
    pp.gsz = 1;
    // causal on a linear cache: CTA lengths grow with the tile, so all heads' longest go first
    pp.hfirst = (a.win == 0 && a.hi == nullptr) ? 1 : 0;
    const dim3 grid(pp.nqt, a.hq);
    prompt_d256_kernel<NP><<<grid, kThreads, C::SMEM, s>>>(pp);
    return cudaGetLastError();
}

template <int NP>
cudaError_t set_d256_attr() {
    return cudaFuncSetAttribute(prompt_d256_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                WideCfg<NP>::SMEM);
}

}  // namespace

}  // namespace wa
