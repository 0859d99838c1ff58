// wa_prompt_pair.cuh — the prompt kernel at head dim 128 with one or two P parts: two 128-row
// query tiles per CTA over shared key tiles.
//
// What it computes is the prompt form of wa_prompt_kernel.cuh (TensorFold pull request #1123,
// "What this changes": bullets "Prompt", "Window.p32", "promptRows(..., hi)", "Scale is a
// parameter"): key tiles of T = 128 keys at absolute positions, each folded into a row's running
// softmax once, fp32 probabilities, P entering P.V as bf16(P) or bf16(P) + bf16(P - bf16(P)).
// A row's arithmetic is its own (one thread owns a whole row), so its bits do not depend on the
// rows it shares a CTA with or on where a prompt is cut.
//
// GB300 layout (one CTA per 256 rows of one query head; tiles q = 0, 1 of 128 rows each):
//   tensor memory   S0 [0, 128)  S1 [128, 256)  O0 [256, 384)  O1 [384, 512)  (fp32 columns)
//                   P of tile q is written over S of tile q: keys [64 h, 64 h + 64) of part k
//                   at column 64 h + 32 k, two bf16 per column.
//   shared memory   Q0, Q1 (32 KiB each), K and V in two stages of 32 KiB each.
//   warp 0          TMA producer: Q0 and Q1 once, then K and V tiles (128-byte swizzle);
//                   tiles that wrap around the ring are copied by the warp with the same swizzle.
//   warp 1          allocates tensor memory; lane 0 issues, per key tile j,
//                     S0(j) = Q0 K(j)^T, O1 += P1(j-1) V(j-1), S1(j) = Q1 K(j)^T, O0 += P0(j) V(j)
//                   so the softmax of one tile runs while the tensor core works for the other.
//                   S0(j) overwrites P0(j-1), which O0 += P0(j-1) V(j-1) read; the tensor core
//                   runs one thread's tcgen05.mma operations in issue order.
//   warp 2          zeroes V rows outside the CTA's key union in the first and last tile.
//   warps 4..7      tile 0, warps 8..11 tile 1: one row per thread (= tensor-memory lane) and
//                   all 128 keys of a tile: the row max over the whole S row, then per 64-key
//                   half mask, scale, exponentials and P into tensor memory; lazy online softmax,
//                   O rescale, epilogue.
// Every wait is bounded (a status bit after kWaitLimitNs) and warp-uniform where a warp waits.
#pragma once

#include "wa_prompt_kernel.cuh"

namespace wa {

namespace {

constexpr int kPairRows = 256;     // query rows per CTA (two tensor-memory tiles of 128)

template <int NP>
struct PairCfg {
    static constexpr int D = 128, T = 128, KB = 2;
    static constexpr int Q_BLOCK = kBM * 128;                  // one 64-dim block of a Q tile
    static constexpr int Q_BYTES = KB * Q_BLOCK;                // one Q tile
    static constexpr int KV_BLOCK = T * 128;
    static constexpr int KV_BYTES = KB * KV_BLOCK;
    static constexpr int OFF_Q = 0;                             // Q0, Q1
    static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;           // 2 stages
    static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;          // 2 stages
    static constexpr int OFF_BAR = OFF_V + 2 * KV_BYTES;
    static constexpr int NBAR = 24;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;         // tmem base, per-warp union bounds
    static constexpr int SMEM = OFF_MISC + 128;
    static constexpr int TMEM_COLS = 512;
    __host__ __device__ static constexpr int s_col(int q) { return q * T; }
    __host__ __device__ static constexpr int o_col(int q) { return 2 * T + q * D; }
    static_assert(NP == 1 || NP == 2, "P parts over S: 32 columns per 64 keys each");
    static_assert(o_col(1) + D <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// barrier indices ([s] = per stage = tile & 1; [q][s] at q * 2 + s; PFULL per query tile).
// A parity wait for phase k is only sound while phase k + 1 cannot have completed: S-done and
// P.V-done are per stage, so the phase after the one the producer waits for (the tile two later)
// needs the very load the producer has not issued yet.
// PHALF[q]: P of the tile's first 64 keys is in tensor memory; PFULL[q]: all of P is.
enum : int {
    PB_Q = 0, PB_KFULL = 1, PB_VFULL = 3, PB_VREADY = 5, PB_SFULL = 7, PB_PFULL = 11, PB_PVDONE = 13,
    PB_DRAIN = 17, PB_PHALF = 18
};

template <int NP>
__global__ void __launch_bounds__(kThreads, 1) prompt_pair_kernel(const __grid_constant__ PromptParams p) {
    using C = PairCfg<NP>;
    constexpr int D = C::D, T = C::T;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {   // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(p.status, WA_STATUS_LAYOUT);
        return;
    }
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);   // [0] tmem base, [1..8] lo, [9..16] hi

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = p.nqt - 1 - static_cast<int>(blockIdx.x);            // longest (causal) tiles first
    const int h = static_cast<int>(blockIdx.y);
    const int g = h / (p.hq / p.hkv);
    const int m0 = qt * kPairRows;

    if (threadIdx.x == 0) {
        mbar_init(BAR(PB_Q), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(PB_KFULL + s), 1);
            mbar_init(BAR(PB_VFULL + s), 1);
            mbar_init(BAR(PB_VREADY + s), 1);
            mbar_init(BAR(PB_PFULL + s), 4);     // [q]: one arrival per softmax warp of the tile
            mbar_init(BAR(PB_PHALF + s), 4);
        }
        for (int qs = 0; qs < 4; ++qs) {
            mbar_init(BAR(PB_SFULL + qs), 1);    // [q][s]: MMA commits
            mbar_init(BAR(PB_PVDONE + qs), 1);
        }
        mbar_init(BAR(PB_DRAIN), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), C::TMEM_COLS);
        tmem_relinquish();
    }

    // softmax threads: tile q, row r of the tile (= tensor-memory lane), row i sees [row_lo, row_hi]
    const int q = warp >= 8 ? 1 : 0;
    const int r = (warp & 3) * 32 + lane;
    const int i = m0 + q * kBM + r;
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
                    atomicOr(p.status, WA_STATUS_BAD_HI);
                    hv = min(max(hv, P), p.p0 + p.n - 1);
                }
            }
            row_hi = hv;
        }
        int mn = lane_ok ? row_lo : INT_MAX, mx = lane_ok ? row_hi : INT_MIN;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
            mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        }
        if (lane == 0) {
            misc[1 + warp - 4] = static_cast<uint32_t>(mn);
            misc[9 + warp - 4] = static_cast<uint32_t>(mx);
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
        // only the query tiles that hold a row: a box wholly past the last row is not loaded
        // (tile 1's rows are then all idle and masked, whatever its shared memory holds)
        const int nq = m0 + kBM < p.n ? 2 : 1;
        mbar_arrive_expect_tx(BAR(PB_Q), nq * C::Q_BYTES);
        for (int t = 0; t < nq; ++t)
            for (int b = 0; b < C::KB; ++b)
                tma_load_3d(sbase + C::OFF_Q + t * C::Q_BYTES + b * C::Q_BLOCK, &p.tq, b * 64, h, m0 + t * kBM,
                            BAR(PB_Q), policy_evict_first());
    }
    int ulo = INT_MAX, uhi = INT_MIN;
    for (int w = 0; w < 8; ++w) {
        ulo = min(ulo, static_cast<int>(misc[1 + w]));
        uhi = max(uhi, static_cast<int>(misc[9 + w]));
    }
    // Key tiles j0..j1 (absolute positions [jT, jT + T)) cover every row's range.
    const int j0 = ulo / T;
    const int ntiles = uhi / T - j0 + 1;   // >= 1: the CTA's first row exists (m0 < n)

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        const uint64_t pol_kv = policy_evict_last();
        bool ok = true;
        int issued = 0;
        for (int idx = 0; idx < ntiles && ok; ++idx) {
            const int s = idx & 1;
            const int key0 = (j0 + idx) * T;
            const int slot0 = p.win > 0 ? key0 % p.ring : key0;
            const bool wrapped = p.win > 0 && slot0 + T > p.ring;
            for (int kv = 0; kv < 2 && ok; ++kv) {
                const uint32_t full = BAR((kv ? PB_VFULL : PB_KFULL) + s);
                const uint32_t dst = sbase + (kv ? C::OFF_V : C::OFF_K) + s * C::KV_BYTES;
                // a stage is free once the last product that read it is done: S1 of tile idx - 2 for
                // K, O1 += P1 V of tile idx - 2 for V (each commit covers every earlier product)
                if (idx >= 2 && !warp_wait(BAR((kv ? PB_PVDONE : PB_SFULL) + 2 + s), ((idx >> 1) - 1) & 1, p.status)) {
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
            mbar_wait(BAR(PB_Q), 0, p.status);
            for (int idx = max(0, issued - 2); idx < issued; ++idx) {
                mbar_wait(BAR(PB_KFULL + (idx & 1)), (idx >> 1) & 1, p.status);
                mbar_wait(BAR(PB_VFULL + (idx & 1)), (idx >> 1) & 1, p.status);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (one thread)
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(kBM, T, 0, 0, p.neg ? 1u : 0u);
            constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
            const uint64_t aq0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
            const uint64_t aq1 = sdesc_sw128(sbase + C::OFF_Q + C::Q_BYTES, 16, 1024);
            auto issue_s = [&](int t, int tile, uint64_t aq, uint64_t bk) {
                const uint32_t d_s = tbase + C::s_col(t);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_bf16_ss(d_s, aq + (((kk >> 2) * C::Q_BLOCK + (kk & 3) * 32) >> 4),
                                bk + (((kk >> 2) * C::KV_BLOCK + (kk & 3) * 32) >> 4), idS, kk > 0 ? 1u : 0u);
                mma_commit(BAR(PB_SFULL + 2 * t + (tile & 1)));
            };
            // O(t) += P(t) V over the keys of one 64-key half of the tile (K steps 4 hh .. 4 hh + 3),
            // every P part; the second half's products are followed by the P.V-done commit.
            auto issue_pv_half = [&](int t, int tile, int hh) {
                const uint64_t v0 = sdesc_sw128(sbase + C::OFF_V + (tile & 1) * C::KV_BYTES, C::KV_BLOCK, 1024);
#pragma unroll
                for (int part = 0; part < NP; ++part)
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const int kk = 4 * hh + k4;
                        mma_bf16_ts(tbase + C::o_col(t), tbase + C::s_col(t) + hh * 64 + part * 32 + k4 * 8,
                                    v0 + ((kk * 16 * 128) >> 4), idO, (tile > 0 || kk > 0 || part > 0) ? 1u : 0u);
                    }
                if (hh == 1) mma_commit(BAR(PB_PVDONE + 2 * t + (tile & 1)));
            };
            // P.V of a tile in two halves: the first 64 keys' products start while the softmax
            // still works on the second 64, which shortens each query tile's S -> softmax -> P.V
            // chain by a half P.V.
            auto issue_pv = [&](int t, int tile) -> bool {
                if (!mbar_wait(BAR(PB_PHALF + t), tile & 1, p.status)) return false;
                tc_fence_after();
                issue_pv_half(t, tile, 0);
                if (!mbar_wait(BAR(PB_PFULL + t), tile & 1, p.status)) return false;
                tc_fence_after();
                issue_pv_half(t, tile, 1);
                return true;
            };
            // The waits for K(j + 1) and V(j) come before the wait for P0(j): both are in shared
            // memory long before the softmax of tile j is done, so once P0(j) is there nothing
            // stands between O0 += P0(j) V(j) and S0(j + 1).
            bool ok = mbar_wait(BAR(PB_Q), 0, p.status) && mbar_wait(BAR(PB_KFULL), 0, p.status);
            for (int j = 0; ok && j < ntiles; ++j) {
                const int s = j & 1, u = j >> 1;
                tc_fence_after();
                const uint64_t bk = sdesc_sw128(sbase + C::OFF_K + s * C::KV_BYTES, 16, 1024);
                issue_s(0, j, aq0, bk);
                if (j >= 1 && !(ok = issue_pv(1, j - 1))) break;
                issue_s(1, j, aq1, bk);
                ok = mbar_wait(BAR(PB_VREADY + s), u & 1, p.status);
                if (ok && j + 1 < ntiles) ok = mbar_wait(BAR(PB_KFULL + (s ^ 1)), ((j + 1) >> 1) & 1, p.status);
                if (ok) ok = issue_pv(0, j);
            }
            if (ok) ok = issue_pv(1, ntiles - 1);
            // every MMA issued so far has finished before tensor memory can be released
            mma_commit(BAR(PB_DRAIN));
            mbar_wait(BAR(PB_DRAIN), 0, p.status);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------ V rows outside the key union -> 0
        for (int idx = 0; idx < ntiles; ++idx) {
            const int s = idx & 1, u = idx >> 1;
            if (!warp_wait(BAR(PB_VFULL + s), u & 1, p.status)) break;
            const int key0 = (j0 + idx) * T;
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
            if (lane == 0) mbar_arrive(BAR(PB_VREADY + s));
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ softmax: tile q, row r, all T columns
        const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t t_s = tbase + lane_addr + C::s_col(q);
        const uint32_t t_o = tbase + lane_addr + C::o_col(q);
        const float c = p.c;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; ok && j < ntiles; ++j) {
            if (!warp_wait(BAR(PB_SFULL + 2 * q + (j & 1)), (j >> 1) & 1, p.status)) { ok = false; break; }
            tc_fence_after();
            // visible columns [vlo, vhi]; interior tiles need no mask at all
            const int kbase = (j0 + j) * T;
            const int vlo = row_lo - kbase, vhi = row_hi - kbase;
            const bool masked = !__all_sync(0xFFFFFFFFu, vlo <= 0 && vhi >= T - 1);
            // pass 1: the tile's row max, over two 64-column loads
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t raw[64];
                tmem_ld64_wait(t_s + half * 64, raw);
                if (masked) {
#pragma unroll
                    for (int k = 0; k < 64; ++k) {
                        const int col = half * 64 + k;
                        mx8[k & 7] = fmaxf(mx8[k & 7], (col >= vlo && col <= vhi) ? __uint_as_float(raw[k]) : -INFINITY);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 64; k += 2)
                        mx8[(k >> 1) & 7] = max3(mx8[(k >> 1) & 7], __uint_as_float(raw[k]), __uint_as_float(raw[k + 1]));
                }
            }
            const float mraw = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                     fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float mt = mraw * c;                       // tile max in log2 units
            // lazy rescale: keep the running max unless the tile's exceeds it by more than kLazy
            const float m_new = (mt > m_run + kLazy) ? mt : m_run;
            const float alpha = (m_new == m_run) ? 1.f : ex2(m_run - m_new);
            const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;

            // an O rescale waits for the previous tile's P.V of this query tile
            if (j >= 1 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
                if (!warp_wait(BAR(PB_PVDONE + 2 * q + ((j - 1) & 1)), ((j - 1) >> 1) & 1, p.status)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32_wait(t_o + cc * 32, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(t_o + cc * 32, o);
                }
            }
            // pass 2, per 64-key half: p = 2^(S c - m_sub), the row sum, and P over the half's own S
            // columns (already read): part k of keys [64 half, 64 half + 64) at column
            // 64 half + 32 k, two bf16 per column.  The residual p - hi is exact in fp32.
            float ls8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) ls8[e] = 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float sv[64];
                {
                    uint32_t raw[64];
                    tmem_ld64_wait(t_s + half * 64, raw);
#pragma unroll
                    for (int e = 0; e < 64; ++e) sv[e] = __uint_as_float(raw[e]);
                }
                if (masked) {   // a masked column is 0 whatever its score (also for scale 0 or a NaN key)
#pragma unroll
                    for (int k = 0; k < 64; ++k) {
                        const int col = half * 64 + k;
                        const float pk = (col >= vlo && col <= vhi) ? ex2(fmaf(sv[k], c, -m_sub)) : 0.f;
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
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t w[NP][16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float a = sv[cc * 32 + 2 * e], b = sv[cc * 32 + 2 * e + 1];
#pragma unroll
                        for (int part = 0; part < NP; ++part) {
                            w[part][e] = pack_bf16(a, b);
                            a -= __uint_as_float(w[part][e] << 16);
                            b -= __uint_as_float(w[part][e] & 0xFFFF0000u);
                        }
                    }
#pragma unroll
                    for (int part = 0; part < NP; ++part) tmem_st16(t_s + half * 64 + part * 32 + cc * 16, w[part]);
                }
                if (half == 0) {   // the first half's P (and any O rescale above) is in place
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(PB_PHALF + q));
                }
            }
            const float lsum = ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
            l_run = (alpha == 1.f) ? (l_run + lsum) : fmaf(l_run, alpha, lsum);
            m_run = m_new;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(PB_PFULL + q));
        }
        // epilogue: o = O / l, bf16; a non-finite row goes to the float64 re-run
        if (ok) ok = warp_wait(BAR(PB_PVDONE + 2 * q + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, p.status);
        if (ok) {
            tc_fence_after();
            bool bad = false;
            uint16_t* orow = p.out + static_cast<int64_t>(i) * p.o_tok + static_cast<int64_t>(h) * D;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32_wait(t_o + cc * 32, o);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float a = __fdiv_rn(__uint_as_float(o[2 * e]), l_run);
                    const float b = __fdiv_rn(__uint_as_float(o[2 * e + 1]), l_run);
                    bad |= !(isfinite(a) && isfinite(b));
                    pk[e] = pack_bf16(a, b);
                }
                if (lane_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            if (lane_ok && bad) p.flags[atomicAdd(p.nflag, 1)] = i * p.hq + h;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, C::TMEM_COLS);
}

template <int NP>
cudaError_t launch_pair(const PromptArgs& a, cudaStream_t s) {
    using C = PairCfg<NP>;
    PromptParams pp{};
    if (!encode_3d(&pp.tq, a.q, C::D, a.hq, a.n, a.q_tok, kBM) ||
        !encode_3d(&pp.tk, a.k, C::D, a.hkv, a.ring, a.k_tok, C::T) ||
        !encode_3d(&pp.tv, a.v, C::D, a.hkv, a.ring, a.v_tok, C::T))
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
    pp.nqt = (a.n + kPairRows - 1) / kPairRows;
    pp.neg = a.scale < 0.f ? 1 : 0;
    pp.c = (a.scale < 0.f ? -a.scale : a.scale) * 1.4426950408889634f;
    pp.gsz = 1;
    const dim3 grid(pp.nqt, a.hq);
    prompt_pair_kernel<NP><<<grid, kThreads, C::SMEM, s>>>(pp);
    return cudaGetLastError();
}

template <int NP>
cudaError_t set_pair_attr() {
    return cudaFuncSetAttribute(prompt_pair_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PairCfg<NP>::SMEM);
}

}  // namespace

}  // namespace wa
