// wa_decode_tc.cu — decode partials on the tensor cores, for large query-head groups.
//
// Same arithmetic contract as decode_part_kernel (TensorFold pull request #1123,
// section "What this changes", bullet "Decode": 256-key chunks at absolute key
// positions, a chunk's (m_c, l_c, o_c) in fp32 with fp32 probabilities, chunks
// with none of the row's keys skipped), for groups of query heads per key head
// large enough (the pages allow up to 16) that scoring on CUDA cores, not HBM,
// bounds the CUDA-core kernel.
//
// GB300 design.  A persistent grid, one CTA per SM, that streams the K and V of
// its units (row, key head, chunk) through shared-memory rings without a break
// between units.  Units come from a counter in the workspace header, long ones
// first: each CTA's producer warp sorts the rows by chunk count (a counting sort
// in shared memory) and walks "levels" from the last: level e holds, for every
// row with more than e chunks, the chunk e places from its end, where the order
// from the end is last chunk, first chunk, then the middle ones.  Whole chunks go
// first, the ragged first and last chunks last, and no empty chunk is taken
// (calls too large for the sort take units in a plain stride).  The producer
// hands each unit, fully described, to the other warps through a ring of unit
// slots, so no other role reads the positions.  160 threads:
//   warp 0  softmax, one lane per query head of the group (tensor-memory lane
//           h = head h; M = 128 with the lanes past the group unused): an
//           online softmax over the chunk's 64-key sub-tiles at absolute
//           positions, probabilities fp32 entering P V as
//           bf16(P) + bf16(P - bf16(P)) from tensor memory; writes m_c, l_c.
//   warp 1  allocates tensor memory; lane 0 issues tcgen05.mma:
//           S = Q K^T (A = Q from tensor memory, B = K, 128-byte swizzle) and
//           O += P V (A = P from tensor memory, B = V read MN-major).
//   warp 2  takes units and publishes them; TMA producer: K and V sub-tiles
//           through rings of stages; a sub-tile that wraps around the ring is
//           copied by the warp with the same swizzle.
//   warp 3  zeroes V rows outside the row's window, so a stale ring slot
//           never meets a zero probability as 0 * inf.
//   warp 4  stages each unit's G query heads into tensor memory (negated for
//           a negative scale, so S carries the sign and the exponent uses
//           |scale|) and copies O of the finished unit into its record.
// The record (m_c in natural-log units, l_c, o_c) is the one the ordered
// merge kernel reads, so the merge and the float64 re-run are shared.  Every
// unit's arithmetic depends only on the unit, so results do not depend on the
// batch, the grid or which CTA took the unit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "wa_internal.h"
#include "wa_ptx.cuh"

namespace wa {

namespace {

constexpr int kSub = 64;            // keys per sub-tile
constexpr int kTcThreads = 160;
constexpr int kUnitSlots = 8;       // unit slots: published units not yet taken by every role
constexpr int kUnitAhead = 4;       // units the producer publishes beyond the one it loads
constexpr int kPlanRows = 2048;     // the sorted schedule serves calls up to this many rows ...
constexpr int kPlanChunks = 1024;   // ... and chunks a row; larger calls take units in a plain stride
constexpr float kLazyTc = 8.0f;     // log2 units the running max may trail before O is rescaled

struct TcParams {
    CUtensorMap tk, tv;           // [rows][ring][hkv][d] rings, box 64 x 1 x 64 x 1, 128-byte swizzle
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* pos;
    float* part;
    int* status;
    int* next_unit;               // zeroed with the workspace header every call
    int rows, hq, hkv, gsize, win, ring, cmax;
    float c;                      // |scale| * log2(e)
    uint32_t qsign;               // 0x80008000 when scale < 0
};

template <int D>
struct TcCfg {
    static constexpr int KB = D / 64;
    static constexpr int KV_BLOCK = kSub * 128;
    static constexpr int KV_BYTES = KB * KV_BLOCK;
    static constexpr int NSK = D == 256 ? 3 : 6, NSV = NSK;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + NSK * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + NSV * KV_BYTES;
    static constexpr int B_KFULL = 0;
    static constexpr int B_KFREE = B_KFULL + NSK;
    static constexpr int B_VFULL = B_KFREE + NSK;
    static constexpr int B_VREADY = B_VFULL + NSV;
    static constexpr int B_VFREE = B_VREADY + NSV;
    static constexpr int B_QT = B_VFREE + NSV;     // Q of a unit in tensor memory
    static constexpr int B_QFREE = B_QT + 1;       // last S of a unit done
    static constexpr int B_SFULL = B_QFREE + 1;
    static constexpr int B_SFREE = B_SFULL + 1;
    static constexpr int B_PFULL = B_SFREE + 1;
    static constexpr int B_PVDONE = B_PFULL + 1;
    static constexpr int B_ODONE = B_PVDONE + 1;   // last P V of a unit done
    static constexpr int B_OFREE = B_ODONE + 1;    // O of a unit copied out
    static constexpr int B_DRAIN = B_OFREE + 1;
    static constexpr int B_UFULL = B_DRAIN + 1;    // [NU] a unit published in the slot
    static constexpr int B_UFREE = B_UFULL + kUnitSlots;   // [NU] the slot read by the 4 other roles
    static constexpr int NBAR = B_UFREE + kUnitSlots;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;    // [0] tensor-memory base
    static constexpr int OFF_RING = OFF_MISC + 16;         // kUnitSlots units (8 ints each)
    static constexpr int OFF_PERM = OFF_RING + 32 * kUnitSlots;  // kPlanRows: row | chunks << 16, by chunks, descending
    static constexpr int OFF_POS = OFF_PERM + 4 * kPlanRows;     // kPlanRows: clamped positions
    static constexpr int OFF_CUR = OFF_POS + 4 * kPlanRows;      // kPlanChunks + 1: histogram, then sort cursors
    static constexpr int OFF_ACC = OFF_CUR + 4 * (kPlanChunks + 1);     // kPlanChunks: rows in level 0, 1, ...
    static constexpr int OFF_START = OFF_ACC + 4 * kPlanChunks;          // kPlanChunks + 1: first unit of each level
    static constexpr int SMEM = OFF_START + 4 * (kPlanChunks + 1);
    // tensor memory: O (D columns), S (64), P hi and lo (2 x 32), Q (D / 2)
    static constexpr int O_COL = 0;
    static constexpr int S_COL = D;
    static constexpr int P_COL = D + kSub;
    static constexpr int Q_COL = D + 2 * kSub;
    static constexpr int TMEM_COLS = 512;
    static_assert(Q_COL + D / 2 <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

// One unit of work: the keys of chunk c (absolute positions [256c, 256c + 255])
// that row r sees through key head g, as sub-tiles t0 .. t0 + nt - 1.
struct Unit {
    int r, g, ci, cbase, kb, ke, t0, nt;
};

// A decode position as the kernels use it: out-of-range positions clamped (the caller reports).
__device__ __forceinline__ int clamp_pos(const TcParams& p, int pp) {
    return (pp < 0 || (p.win == 0 && pp >= p.ring)) ? (pp < 0 ? 0 : p.ring - 1) : pp;
}

// Fills x for row r, key head g and chunk ci of a row at clamped position pp; false when the
// chunk holds none of the row's keys.
__device__ __forceinline__ bool unit_from(const TcParams& p, int r, int g, int ci, int pp, Unit& x) {
    x.r = r;
    x.g = g;
    x.ci = ci;
    const int lo = p.win > 0 ? max(0, pp - p.win + 1) : 0;
    const int c = lo / kChunk + ci;
    if (c > pp / kChunk) return false;
    x.cbase = c * kChunk;
    x.kb = max(lo, x.cbase);
    x.ke = min(pp, x.cbase + kChunk - 1);
    x.t0 = (x.kb - x.cbase) / kSub;
    x.nt = (x.ke - x.cbase) / kSub - x.t0 + 1;
    return true;
}

// The same for unit index u = (r * hkv + g) * cmax + ci, reading the row's position (reported once
// per row, by its unit (r, 0, 0), when out of range).
__device__ __forceinline__ bool unit_at(const TcParams& p, int u, Unit& x, bool report) {
    const int ci = u % p.cmax, rg = u / p.cmax;
    const int g = rg % p.hkv, r = rg / p.hkv;
    const int raw = p.pos[r];
    const int pp = clamp_pos(p, raw);
    if (report && pp != raw && ci == 0 && g == 0) atomicOr(p.status, WA_STATUS_BAD_POS);
    return unit_from(p, r, g, ci, pp, x);
}

// Chunks holding any of a row's keys (at least 1) at clamped position pp.
__device__ __forceinline__ int chunks_at(const TcParams& p, int pp) {
    const int lo = p.win > 0 ? max(0, pp - p.win + 1) : 0;
    return min(p.cmax, pp / kChunk - lo / kChunk + 1);
}

// Inclusive sum over the warp's lanes.
__device__ __forceinline__ int warp_scan_incl(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_kernel(const __grid_constant__ TcParams p) {
    using C = TcCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.status, WA_STATUS_LAYOUT);
        return;
    }
    const int units = p.rows * p.hkv * p.cmax;
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NBAR; ++i) mbar_init(BAR(i), (i >= C::B_UFREE && i < C::B_UFREE + kUnitSlots) ? 4 : 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = misc[0];
    volatile int* uring = reinterpret_cast<volatile int*>(smem + C::OFF_RING);   // 8 ints a slot

    // Every role but the producer: the U-th published unit (x.nt = 0 after the last).  The MMA
    // role runs on one thread (whole = false), the others as a warp; each role arrives once.
    auto take_unit = [&](int U, Unit& x, bool whole) -> bool {
        const int sl = U % kUnitSlots;
        const uint32_t ph = static_cast<uint32_t>(U / kUnitSlots) & 1u;
        if (!(whole ? warp_wait(BAR(C::B_UFULL + sl), ph, p.status) : mbar_wait(BAR(C::B_UFULL + sl), ph, p.status)))
            return false;
        volatile int* e = uring + 8 * sl;
        x.r = e[0]; x.g = e[1]; x.ci = e[2]; x.cbase = e[3];
        x.kb = e[4]; x.ke = e[5]; x.t0 = e[6]; x.nt = e[7];
        if (whole) __syncwarp();
        if (!whole || lane == 0) mbar_arrive(BAR(C::B_UFREE + sl));
        return true;
    };

    if (warp == 2) {
        // ------------------------------------------------ unit schedule; TMA producer: K then V of each sub-tile
        const uint64_t pol = policy_evict_first();
        if (lane == 0) {
            prefetch_tensormap(&p.tk);
            prefetch_tensormap(&p.tv);
        }
        uint32_t* perm = reinterpret_cast<uint32_t*>(smem + C::OFF_PERM);
        int* spos = reinterpret_cast<int*>(smem + C::OFF_POS);
        int* cur = reinterpret_cast<int*>(smem + C::OFF_CUR);
        int* acc = reinterpret_cast<int*>(smem + C::OFF_ACC);
        int* start = reinterpret_cast<int*>(smem + C::OFF_START);
        const int cm = p.cmax;
        const bool planned = p.rows <= kPlanRows && cm <= kPlanChunks;
        int total = 0;
        if (planned) {
            // rows sorted by chunk count, descending (counting sort)
            for (int c = lane; c <= cm; c += 32) cur[c] = 0;
            __syncwarp();
            for (int r = lane; r < p.rows; r += 32) {
                const int raw = p.pos[r];
                const int pp = clamp_pos(p, raw);
                if (pp != raw && blockIdx.x == 0) atomicOr(p.status, WA_STATUS_BAD_POS);
                spos[r] = pp;
                atomicAdd(&cur[chunks_at(p, pp)], 1);
            }
            __syncwarp();
            // level l takes the chunk e = cm - 1 - l places from each row's end; acc[l] = rows with more than e chunks
            int carry = 0;
            for (int b = 0; b < cm; b += 32) {
                const int i = b + lane;
                const int v = warp_scan_incl(i < cm ? cur[cm - i] : 0, lane) + carry;
                if (i < cm) acc[i] = v;
                carry = __shfl_sync(0xFFFFFFFFu, v, 31);
            }
            __syncwarp();
            // start[l] = units before level l (hkv units per row of a level)
            carry = 0;
            for (int b = 0; b < cm; b += 32) {
                const int i = b + lane;
                const int a = i < cm ? acc[i] : 0;
                const int v = warp_scan_incl(a, lane);
                if (i < cm) start[i] = p.hkv * (carry + v - a);
                carry += __shfl_sync(0xFFFFFFFFu, v, 31);
            }
            if (lane == 0) start[cm] = p.hkv * carry;
            // rows with n chunks go after every row with more
            for (int c = lane; c <= cm; c += 32) cur[c] = c >= cm ? 0 : acc[cm - 1 - c];
            __syncwarp();
            for (int r = lane; r < p.rows; r += 32) {
                const int n = chunks_at(p, spos[r]);
                perm[atomicAdd(&cur[n], 1)] = static_cast<uint32_t>(r) | (static_cast<uint32_t>(n) << 16);
            }
            __syncwarp();
            total = start[cm];
        }
        // unit k of the schedule: the row's chunks from its end are last, first, then the middle ones
        auto unit_of = [&](int k, Unit& x) {
            int lo = 0, hi = cm - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (start[mid] <= k) lo = mid; else hi = mid - 1;
            }
            const int e = cm - 1 - lo, j = k - start[lo];
            const uint32_t ent = perm[j / p.hkv];
            const int r = static_cast<int>(ent & 0xFFFFu), n = static_cast<int>(ent >> 16), g = j % p.hkv;
            const int rank = n - 1 - e;
            const int ci = rank == n - 1 ? n - 1 : (rank == n - 2 ? 0 : rank + 1);
            unit_from(p, r, g, ci, spos[r], x);
        };
        // The next unit (x.nt = 0 once there is none).  A CTA's first unit is its index; each later
        // one comes from the counter, asked one unit ahead so its answer is back before it is
        // needed.  Without a schedule: a plain stride, skipping empty chunks.
        int k_cur = blockIdx.x, k_ans = 0, su = blockIdx.x;
        bool asked = false;
        auto next_unit = [&](Unit& x) {
            x = Unit{};
            if (planned) {
                if (asked) k_cur = __shfl_sync(0xFFFFFFFFu, k_ans, 0) + static_cast<int>(gridDim.x);
                if (k_cur >= total) return;
                if (lane == 0) k_ans = atomicAdd(p.next_unit, 1);
                asked = true;
                unit_of(k_cur, x);
                return;
            }
            for (; su < units; su += gridDim.x)
                if (unit_at(p, su, x, lane == 0)) {
                    su += gridDim.x;
                    return;
                }
            x = Unit{};
        };
        int Upub = 0;
        auto publish = [&](const Unit& x) -> bool {
            const int sl = Upub % kUnitSlots;
            if (Upub >= kUnitSlots &&
                !warp_wait(BAR(C::B_UFREE + sl), static_cast<uint32_t>(Upub / kUnitSlots - 1) & 1u, p.status))
                return false;
            if (lane == 0) {
                volatile int* e = uring + 8 * sl;
                e[0] = x.r; e[1] = x.g; e[2] = x.ci; e[3] = x.cbase;
                e[4] = x.kb; e[5] = x.ke; e[6] = x.t0; e[7] = x.nt;
                mbar_arrive(BAR(C::B_UFULL + sl));
            }
            __syncwarp();
            ++Upub;
            return true;
        };
        // publish the next unit, or the end marker once (x.nt = 0)
        bool ended = false;
        auto publish_next = [&]() -> bool {
            if (ended) return true;
            Unit x;
            next_unit(x);
            ended = x.nt <= 0;
            return publish(x);
        };
        const size_t row_elems = static_cast<size_t>(p.ring) * p.hkv * D;
        bool ok = true;
        int issued[2] = {0, 0};
        int T = 0;
        // The producer keeps kUnitAhead units published beyond the one it loads, so every role
        // knows its next unit (and the Q/O warp can fetch its queries) well before it starts.
        for (int l = 0; l < kUnitAhead && ok; ++l) ok = publish_next();
        for (int U = 0; ok; ++U) {
            Unit x;
            {
                volatile int* e = uring + 8 * (U % kUnitSlots);   // published by this warp
                x.r = e[0]; x.g = e[1]; x.ci = e[2]; x.cbase = e[3];
                x.kb = e[4]; x.ke = e[5]; x.t0 = e[6]; x.nt = e[7];
            }
            if (x.nt <= 0) break;
            if (!(ok = publish_next())) break;
            for (int idx = 0; idx < x.nt && ok; ++idx, ++T) {
                const int key0 = x.cbase + (x.t0 + idx) * kSub;
                const int slot0 = key0 % p.ring;
                const bool wrapped = slot0 + kSub > p.ring;
                for (int kv = 0; kv < 2; ++kv) {
                    const int NS = kv ? C::NSV : C::NSK;
                    const int s = T % NS, use = T / NS;
                    const uint32_t full = BAR((kv ? C::B_VFULL : C::B_KFULL) + s);
                    const uint32_t dst = sbase + (kv ? C::OFF_V : C::OFF_K) + s * C::KV_BYTES;
                    if (use > 0 && !warp_wait(BAR((kv ? C::B_VFREE : C::B_KFREE) + s), (use - 1) & 1, p.status)) {
                        ok = false;
                        break;
                    }
                    if (!wrapped) {
                        if (lane == 0) {
                            mbar_arrive_expect_tx(full, C::KV_BYTES);
                            for (int b = 0; b < C::KB; ++b)
                                tma_load_4d(dst + b * C::KV_BLOCK, kv ? &p.tv : &p.tk, b * 64, x.g, slot0, x.r, full,
                                            pol);
                        }
                    } else {
                        // a sub-tile whose slots wrap to the start of the ring: copied by the warp
                        const uint16_t* base = (kv ? p.v : p.k) + static_cast<size_t>(x.r) * row_elems;
                        for (int u16 = lane; u16 < kSub * C::KB * 8; u16 += 32) {
                            const int kr = u16 / (C::KB * 8), rem = u16 % (C::KB * 8);
                            const int b = rem / 8, cc = rem % 8;
                            const int slot = (key0 + kr) % p.ring;
                            const uint4 val =
                                ld_global_nc_v4(base + (static_cast<size_t>(slot) * p.hkv + x.g) * D + b * 64 + cc * 8);
                            st_shared_v4(dst + b * C::KV_BLOCK + kr * 128 + ((cc ^ (kr & 7)) * 16), val.x, val.y, val.z,
                                         val.w);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(full);
                    }
                    __syncwarp();
                    issued[kv] = T + 1;
                }
            }
        }
        // let the copies in flight land before the block exits, whichever role stopped early (after a
        // normal run every one was consumed, and the waits return at once)
        if (lane == 0) {
            for (int t = max(0, issued[0] - C::NSK); t < issued[0]; ++t)
                mbar_wait(BAR(C::B_KFULL + t % C::NSK), (t / C::NSK) & 1, p.status);
            for (int t = max(0, issued[1] - C::NSV); t < issued[1]; ++t)
                mbar_wait(BAR(C::B_VFULL + t % C::NSV), (t / C::NSV) & 1, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer: S(T), then P V(T - 1)
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(128, kSub, 0, 0);
            constexpr uint32_t idO = idesc_bf16_f32(128, D, 0, 1);
            bool ok = true;
            int T = 0, U = 0;
            // the sub-tile whose P V is still to issue
            bool pv_pending = false, pv_first = false, pv_last = false;
            int pv_T = 0, pv_U = 0;
            auto issue_pv = [&]() -> bool {
                const int ps = pv_T % C::NSV, pu = pv_T / C::NSV;
                if (!mbar_wait(BAR(C::B_PFULL), pv_T & 1, p.status)) return false;
                if (!mbar_wait(BAR(C::B_VREADY + ps), pu & 1, p.status)) return false;
                if (pv_first && pv_U > 0 && !mbar_wait(BAR(C::B_OFREE), (pv_U - 1) & 1, p.status)) return false;
                tc_fence_after();
                const uint32_t vst = sbase + C::OFF_V + ps * C::KV_BYTES;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int kk = 0; kk < kSub / 16; ++kk) {
                        const uint64_t b = sdesc_sw128(vst + kk * 16 * 128, C::KV_BLOCK, 1024);
                        mma_bf16_ts(tbase + C::O_COL, tbase + C::P_COL + half * (kSub / 2) + kk * 8, b, idO,
                                    (!pv_first || kk > 0 || half > 0) ? 1u : 0u);
                    }
                }
                mma_commit(BAR(C::B_PVDONE));
                mma_commit(BAR(C::B_VFREE + ps));
                if (pv_last) mma_commit(BAR(C::B_ODONE));
                return true;
            };
            while (ok) {
                Unit x;
                if (!(ok = take_unit(U, x, false)) || x.nt <= 0) break;
                ok = mbar_wait(BAR(C::B_QT), U & 1, p.status);
                for (int idx = 0; idx < x.nt && ok; ++idx, ++T) {
                    const int s = T % C::NSK, use = T / C::NSK;
                    ok = mbar_wait(BAR(C::B_KFULL + s), use & 1, p.status);
                    if (ok && T >= 1) ok = mbar_wait(BAR(C::B_SFREE), (T - 1) & 1, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kst = sbase + C::OFF_K + s * C::KV_BYTES;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t b = sdesc_sw128(kst + (kk >> 2) * C::KV_BLOCK + (kk & 3) * 32, 16, 1024);
                        mma_bf16_ts(tbase + C::S_COL, tbase + C::Q_COL + kk * 8, b, idS, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(BAR(C::B_SFULL));
                    mma_commit(BAR(C::B_KFREE + s));
                    if (idx == x.nt - 1) mma_commit(BAR(C::B_QFREE));
                    if (pv_pending && !(ok = issue_pv())) break;
                    pv_pending = true;
                    pv_first = idx == 0;
                    pv_last = idx == x.nt - 1;
                    pv_T = T;
                    pv_U = U;
                }
                ++U;
            }
            if (ok && pv_pending) issue_pv();
            mma_commit(BAR(C::B_DRAIN));
            mbar_wait(BAR(C::B_DRAIN), 0, p.status);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------ V rows outside [kb, ke] -> 0
        int T = 0;
        bool ok = true;
        for (int U = 0; ok; ++U) {
            Unit x;
            if (!(ok = take_unit(U, x, true)) || x.nt <= 0) break;
            for (int idx = 0; idx < x.nt; ++idx, ++T) {
                const int s = T % C::NSV, use = T / C::NSV;
                if (!warp_wait(BAR(C::B_VFULL + s), use & 1, p.status)) {
                    ok = false;
                    break;
                }
                const int key0 = x.cbase + (x.t0 + idx) * kSub;
                const int z_lo = min(kSub, max(0, x.kb - key0));             // rows [0, z_lo)
                const int z_hi = max(0, min(kSub, x.ke - key0 + 1));          // rows [z_hi, kSub)
                if (z_lo > 0 || z_hi < kSub) {
                    const uint32_t vst = sbase + C::OFF_V + s * C::KV_BYTES;
                    const int nz = z_lo + (kSub - z_hi);
                    for (int u16 = lane; u16 < nz * C::KB * 8; u16 += 32) {
                        const int zr = u16 / (C::KB * 8), rem = u16 % (C::KB * 8);
                        const int row = zr < z_lo ? zr : z_hi + (zr - z_lo);
                        st_shared_v4(vst + (rem / 8) * C::KV_BLOCK + row * 128 + (rem % 8) * 16, 0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(C::B_VREADY + s));
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------ Q of each unit in, O of the previous unit out
        const int h = lane;
        const bool live = h < p.gsize;
        bool ok = true;
        int U = 0;
        float* prev_rec = nullptr;
        // O of a finished unit into its record: up to 128 columns loaded per wait, and O is handed
        // back as soon as the last load has landed, before the last stores
        auto copy_out = [&](float* rec, int Uo) -> bool {
            if (!warp_wait(BAR(C::B_ODONE), Uo & 1, p.status)) return false;
            tc_fence_after();
            constexpr int NB = D >= 128 ? 4 : D / 32;     // 32-column loads per batch
#pragma unroll 1
            for (int cb = 0; cb < D / 32; cb += NB) {
                uint32_t o[NB][32];
#pragma unroll
                for (int b = 0; b < NB; ++b) tmem_ld32(tbase + C::O_COL + (cb + b) * 32, o[b]);
                tmem_wait_ld();
                if (cb + NB >= D / 32) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(BAR(C::B_OFREE));
                }
                if (live) {
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        float4* dst = reinterpret_cast<float4*>(rec + 4 + (cb + b) * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(__uint_as_float(o[b][4 * e]), __uint_as_float(o[b][4 * e + 1]),
                                                 __uint_as_float(o[b][4 * e + 2]), __uint_as_float(o[b][4 * e + 3]));
                    }
                }
            }
            return true;
        };
        while (ok) {
            Unit x;
            if (!(ok = take_unit(U, x, true)) || x.nt <= 0) break;
            const size_t head = static_cast<size_t>(x.r) * p.hq + static_cast<size_t>(x.g) * p.gsize + h;
            const uint4* qrow = reinterpret_cast<const uint4*>(p.q + head * D);
            uint4 qv[D / 8];
#pragma unroll
            for (int e = 0; e < D / 8; ++e) qv[e] = live ? __ldg(qrow + e) : make_uint4(0u, 0u, 0u, 0u);
            if (U > 0 && !warp_wait(BAR(C::B_QFREE), (U - 1) & 1, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < D / 64; ++cb) {       // 64 dims = 32 columns per store
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    w[4 * e] = qv[cb * 8 + e].x ^ p.qsign;
                    w[4 * e + 1] = qv[cb * 8 + e].y ^ p.qsign;
                    w[4 * e + 2] = qv[cb * 8 + e].z ^ p.qsign;
                    w[4 * e + 3] = qv[cb * 8 + e].w ^ p.qsign;
                }
                tmem_st32(tbase + C::Q_COL + cb * 32, w);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::B_QT));
            if (U > 0 && !(ok = copy_out(prev_rec, U - 1))) break;
            prev_rec = p.part + (head * p.cmax + x.ci) * (D + 4);
            ++U;
        }
        if (ok && U > 0) copy_out(prev_rec, U - 1);
    } else {
        // ------------------------------------------------ warp 0: softmax, lane = query head
        const int h = lane;
        const bool live = h < p.gsize;
        const float cl = p.c;
        bool ok = true;
        int T = 0;
        for (int U = 0; ok; ++U) {
            Unit x;
            if (!(ok = take_unit(U, x, true)) || x.nt <= 0) break;
            float m_run = -INFINITY, l_run = 0.f;
            for (int idx = 0; idx < x.nt; ++idx, ++T) {
                if (!warp_wait(BAR(C::B_SFULL), T & 1, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t raw[64];
                tmem_ld64_wait(tbase + C::S_COL, raw);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(C::B_SFREE));
                const int key0 = x.cbase + (x.t0 + idx) * kSub;
                const int vlo = x.kb - key0, vhi = x.ke - key0;   // visible columns [vlo, vhi]
                // eight independent max and sum chains (a chain of 64 would pace the warp)
                float mx8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
                for (int k = 0; k < kSub; ++k)
                    mx8[k & 7] = fmaxf(mx8[k & 7], (k >= vlo && k <= vhi) ? __uint_as_float(raw[k]) : -INFINITY);
                const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                const float mt = mx * cl;
                const float m_new = (mt > m_run + kLazyTc) ? mt : m_run;
                const float alpha = (m_new == m_run) ? 1.f : ex2(m_run - m_new);
                const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
                float pv[kSub];
                float ls8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) ls8[e] = 0.f;
#pragma unroll
                for (int k = 0; k < kSub; ++k) {
                    pv[k] = (k >= vlo && k <= vhi) ? ex2(fmaf(__uint_as_float(raw[k]), cl, -m_sub)) : 0.f;
                    ls8[k & 7] += pv[k];                         // keys k = e mod 8 in key order
                }
                const float ls = ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
                l_run = (alpha == 1.f) ? (l_run + ls) : fmaf(l_run, alpha, ls);
                m_run = m_new;
                // P V of the previous sub-tile must be done before P is overwritten (and O rescaled)
                if (T >= 1) {
                    if (!warp_wait(BAR(C::B_PVDONE), (T - 1) & 1, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (idx > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
#pragma unroll 1
                        for (int cc = 0; cc < D / 32; ++cc) {
                            uint32_t o[32];
                            tmem_ld32_wait(tbase + C::O_COL + cc * 32, o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(tbase + C::O_COL + cc * 32, o);
                        }
                        tmem_wait_st();
                    }
                }
                // P = bf16(p) + bf16(p - bf16(p)) into tensor memory, two bf16 per column
                uint32_t whi[32], wlo[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float a = pv[2 * e], b = pv[2 * e + 1];
                    whi[e] = pack_bf16(a, b);
                    const float ah = __uint_as_float(whi[e] << 16), bh = __uint_as_float(whi[e] & 0xFFFF0000u);
                    wlo[e] = pack_bf16(a - ah, b - bh);
                }
                tmem_st32(tbase + C::P_COL, whi);
                tmem_st32(tbase + C::P_COL + kSub / 2, wlo);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(C::B_PFULL));
            }
            if (ok && live) {
                float* rec = p.part + ((static_cast<size_t>(x.r) * p.hq + static_cast<size_t>(x.g) * p.gsize + h) * p.cmax +
                                       x.ci) * (D + 4);
                rec[0] = m_run * 0.69314718055994531f;   // natural-log units
                rec[1] = l_run;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, C::TMEM_COLS);
}

// [rows, ring, hkv, d] bf16 as a 4-D tensor map with a box of 64 x 1 x 64 x 1 and 128-byte swizzle.
bool encode_ring_sw128(CUtensorMap* m, const void* base, int d, int hkv, int ring, int rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(ring),
                          static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(hkv) * d * 2,
                             static_cast<cuuint64_t>(ring) * hkv * d * 2};
    cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kSub), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

template <int D>
cudaError_t launch_tc_d(const DecodeArgs& a, cudaStream_t s) {
    using C = TcCfg<D>;
    TcParams tp{};
    if (!encode_ring_sw128(&tp.tk, a.k, D, a.hkv, a.ring, a.rows) || !encode_ring_sw128(&tp.tv, a.v, D, a.hkv, a.ring, a.rows))
        return cudaErrorInvalidValue;
    tp.q = static_cast<const uint16_t*>(a.q);
    tp.k = static_cast<const uint16_t*>(a.k);
    tp.v = static_cast<const uint16_t*>(a.v);
    tp.pos = a.pos;
    tp.part = a.part;
    tp.status = &a.hdr->status;
    tp.next_unit = &a.hdr->next_unit;
    tp.rows = a.rows; tp.hq = a.hq; tp.hkv = a.hkv; tp.gsize = a.hq / a.hkv; tp.win = a.win; tp.ring = a.ring;
    tp.cmax = a.cmax;
    tp.qsign = a.scale < 0.f ? 0x80008000u : 0u;
    tp.c = (a.scale < 0.f ? -a.scale : a.scale) * 1.4426950408889634f;
    const int64_t units = static_cast<int64_t>(a.rows) * a.hkv * a.cmax;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = static_cast<int>(units < sms ? units : sms);
    decode_tc_kernel<D><<<grid, kTcThreads, C::SMEM, s>>>(tp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t decode_tc_prepare_device(int) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcCfg<128>::SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<256>::SMEM);
}

cudaError_t launch_decode_tc_part(const DecodeArgs& a, cudaStream_t s) {
    return a.d == 256 ? launch_tc_d<256>(a, s) : launch_tc_d<128>(a, s);
}

}  // namespace wa
