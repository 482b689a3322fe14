// fa_decode.cuh -- split-KV (Flash-Decoding) single-token attention for sm_103a.
//
// What is computed: for each sequence b and query head h, the attention of the single
// query q[b, h] over the cached keys/values [0, kv_lens[b]) of K/V head h / (Hq / Hkv)
// (page "flash-attention-v100", flash_attn_with_kvcache with cache_seqlens; "Changelog",
// "2.2: Optimize for inference").  As the Flash-Decoding steps describe (page
// "flash attention-2 github"): (1) the keys are cut into chunks, (2) each chunk's attention
// is computed independently, writing a partial output and its log-sum-exp, (3) a separate
// kernel merges them with the log-sum-exp weights.
//
// Splitting (page "flash-attention-v100", "Changelog", "2.2" spreads the KV loading over
// several thread blocks without fixing how; this is the reading taken here): the keys of
// every (sequence b, kv head) pair, in 128-key tiles, are laid end to end in the order
// (b, kv head), and CTA c takes the tiles [c W, (c + 1) W).  W is the total divided
// by the grid, so every CTA streams the same number of tiles whatever the length mix,
// but at least ceil(T_max / (num_splits - 1)) for the longest pair's T_max tiles, so no
// pair meets more than num_splits ranges.  A pair cut by range boundaries yields one
// segment per range it meets; each segment is computed independently and writes a
// partial output and its log-sum-exp into the pair's next slot, which the merge kernel
// combines.  The plan is laid over groups of g adjacent kv heads (g = 8, 4 or 2, the
// largest that divides Hkv): a group's tiles count once, and CTAs g r .. g r + g - 1 take
// the same range r, one head each (DecParams::kv_group).  The g streams then read, at
// about the same time, head rows that sit side by side in memory at each key: whole
// DRAM pages are used together, and where a row is not a whole number of 128-byte lines
// (D = 96: 192 bytes) the line two heads share at their common edge is read once.
//
// Split kernel (persistent, one CTA per SM, walking the work items):
//  * the producer warp streams, per item, the Q rows of the query heads sharing the KV head
//    (a 16-row box) and the item's K/V tiles of 128 keys through a 3-stage TMA ring;
//  * the MMA warp computes S^T = K Q^T with the 128 keys of a tile as the M dimension and
//    the query heads (padded to 16) as N, into TMEM, then O^T += V^T P^T with the 128 head
//    dims as M (V read MN-major straight from the swizzled tile, P^T from shared memory);
//  * four compute warps own one key (for S^T) and one head dim (for O^T) each: per tile a
//    cross-warp max per head, exp2 with the scale folded in, a lazily rescaled O^T, and at
//    the end of an item the division by l and the partial (o, lse) store.
// Decode reads every K/V byte exactly once: HBM bandwidth is the roofline.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#pragma once

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

struct DecParams {
    int B, Hq, Hkv, group, Smax, ns;
    float scale_log2;
    const int32_t* kv_lens;
    float* o_part;    // [B, Hq, ns, D]
    float* lse_part;  // [B, Hq, ns]
    int split_grid;   // CTAs of the split kernel (sets the range width)
    // g, the kv heads planned as one entry: range r of the plan over (b, kv heads
    // g k .. g k + g - 1) is streamed for head g k + i by CTA g r + i.
    int kv_group;
    void* o;          // [B, Hq, D]
    float* lse;       // [B, Hq] or null
    int q_rows;  // query-head rows per Q box; rows past q_rows * sq are never read
    // Several query tokens per sequence (flash_attn_with_kvcache with seqlen_q > 1): the
    // MMA's N columns hold (token s, head h) as column s * group + h; with `causal` token s
    // sees keys j <= kv_len - sq + s (bottom-right alignment).  sq = 1 for plain decode.
    int sq, causal;
    // Paged cache (page "flash-attention-v100", flash_attn_with_kvcache block_table;
    // "Changelog", "2.5: Paged KV cache"): key r of sequence b is row r % page_size of
    // page block_table[b * max_pages + r / page_size]; page_size is a multiple of 128.
    const int32_t* block_table;  // null: contiguous [B, Smax, Hkv, D] cache
    int page_size, max_pages;
    int* status;
};

constexpr int kDecBN = 128;  // keys per tile of the split plan
constexpr int kDecMaxB = 1024;
constexpr int kDecMaxKvGroup = 8;  // most kv heads planned as one entry of the split plan
constexpr int kDecThreads = 192;
constexpr int kDecProducerWarp = 4;
constexpr int kDecMmaWarp = 5;
constexpr int kDecMaxBars = 48;

struct DecSmemTail {
    uint64_t bars[kDecMaxBars];
    alignas(16) float red[2][4][16];   // per-tile cross-warp max, double-buffered
    alignas(16) float lred[4][16];     // end-of-item cross-warp sums
    int lens[kDecMaxB];
    int prefix[kDecMaxB + 1];  // exclusive prefix over b of the tiles of one pair of b
    int warp_sums[4];
    int max_len;
    int width;        // W, tiles per CTA range
    int total_tiles;  // (Hkv / kv_group) * prefix[B]
    uint32_t tmem_slot;
    int abort_flag;
};

template <int D_>
struct DecCfg {
    static constexpr int D = D_;
    static constexpr int DA = (D + 63) / 64;        // 128-byte column atoms per row
    // Keys per MMA step (and per ring stage): 64 at D = 256, 256 at D = 64 (a step of 128
    // keys there carries only 32 KB, too little to cover the step's fixed costs: its
    // barrier waits and commits, and the compute warps' cross-warp reduction), else 128.
    static constexpr int SUB = D > 128 ? 64 : (D <= 64 ? 256 : 128);
    static constexpr int KM = SUB >= 128 ? SUB / 128 : 1;  // 128-key M blocks of S^T per step
    static constexpr int BOX = SUB < 128 ? SUB : 128;     // rows of one TMA box
    static constexpr int NBOX = SUB / BOX;                // boxes per column atom per step
    static constexpr int NS = 3;                          // ring stages: 192 KB of K/V in flight
    static constexpr int OM = (D + 127) / 128;      // 128-row blocks of O^T
    static constexpr int KVBytes = SUB * DA * 128;
    static constexpr int QBytes = DA * 16 * 128;
    static constexpr int PBytes = (SUB / 64) * 16 * 128;
    // barrier indices
    static constexpr int BarQFull = 0;                // 2
    static constexpr int BarQEmpty = BarQFull + 2;    // 2
    static constexpr int BarKFull = BarQEmpty + 2;    // NS
    static constexpr int BarKEmpty = BarKFull + NS;
    static constexpr int BarVFull = BarKEmpty + NS;
    static constexpr int BarVEmpty = BarVFull + NS;
    static constexpr int BarSFull = BarVEmpty + NS;   // 2
    // P full and O done: one barrier per P^T buffer.  With P^T double-buffered the compute
    // warps may finish tile j + 1 before the MMA warp has observed tile j; a single barrier
    // would then complete two phases ahead of its waiter and the parity wait would miss one.
    static constexpr int BarPFull = BarSFull + 2;     // 2
    static constexpr int BarODone = BarPFull + 2;     // 2
    static constexpr int BarODrained = BarODone + 2;
    static constexpr int BarFinal = BarODrained + 1;
    static constexpr int NumBars = BarFinal + 1;
    // P^T is double-buffered: the compute warps write tile j's while P.V of tile j-1 reads
    // the other buffer.
    static constexpr int TileBytes = 2 * NS * KVBytes + 2 * QBytes + 2 * PBytes;
    static constexpr int SmemBytes = 1024 + TileBytes + (int)sizeof(DecSmemTail);
    static_assert(NumBars <= kDecMaxBars, "barrier slots");
    static_assert(SmemBytes <= 232448, "decode shared memory budget");
    // TMEM: two S^T slots of KM 16-column blocks each, then the O^T blocks.
    static constexpr int SCols = 16 * KM;
    static constexpr int OCol0 = 2 * SCols;
    static constexpr int TmemCols = OCol0 + 16 * OM <= 64 ? 64 : 128;
    static_assert(OCol0 + 16 * OM <= 128, "TMEM budget");
    static_assert(D % 32 == 0 && D <= 256, "head dim");
};

// MMA steps of SUB keys that cover an item of ntiles 128-key tiles.
template <class DC>
__device__ __forceinline__ int dec_steps(int ntiles) {
    return (ntiles * kDecBN + DC::SUB - 1) / DC::SUB;
}

// One segment of work: keys [k0, k1) of pair (b, hk), written to partial slot c.
struct DecItem {
    int b, hk, c, k0, k1, ntiles;
};

// Width W of the CTA ranges (shared by the split and merge kernels, which must agree).
__device__ __forceinline__ int decode_range_width(int total_tiles, int max_pair_tiles, int grid, int ns) {
    long long w = ((long long)total_tiles + grid - 1) / grid;
    if (ns >= 2)
        w = max(w, ((long long)max_pair_tiles + ns - 2) / (ns - 1));
    else
        w = max(w, (long long)total_tiles);  // one range: no pair is cut
    return (int)max(w, 1LL);
}

// The next segment of range `rng`, starting at tile x (x advances past it).  The plan
// holds Hu = Hkv / kv_group entries per sequence; entry u stands for kv heads
// u * kv_group .. u * kv_group + kv_group - 1, and this CTA computes head u * kv_group + sub.
__device__ __forceinline__ bool next_segment(const DecSmemTail& t, int B, int Hu, int rng, int kv_group,
                                             int sub, int& x, int end, DecItem& it) {
    if (x >= end) return false;
    int lo = 0, hi = B;  // largest b with Hu * prefix[b] <= x; that b has tiles
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (Hu * t.prefix[mid] <= x) lo = mid; else hi = mid;
    }
    const int tb = t.prefix[lo + 1] - t.prefix[lo];
    const int hu = (x - Hu * t.prefix[lo]) / tb;
    const int pstart = Hu * t.prefix[lo] + hu * tb;  // first tile of entry (lo, hu)
    const int seg_end = min(end, pstart + tb);
    it.b = lo;
    it.hk = hu * kv_group + sub;
    it.c = rng - pstart / t.width;  // ranges met by this pair before this one
    it.k0 = (x - pstart) * kDecBN;
    it.k1 = min((seg_end - pstart) * kDecBN, t.lens[lo]);
    it.ntiles = seg_end - x;
    x = seg_end;
    return true;
}

// Shared-memory byte address of P^T[h][key] in the 128-byte-swizzled K-major layout of a
// 16-row x 128-key operand (two 64-key atoms of 16 rows x 128 bytes).
__device__ __forceinline__ uint32_t pt_addr(uint32_t sP, int h, int key) {
    const uint32_t byte = (uint32_t)(key & 63) * 2u;
    return sP + (uint32_t)(key >> 6) * 2048u + (uint32_t)h * 128u +
           ((((byte >> 4) ^ (uint32_t)(h & 7)) << 4) | (byte & 15u));
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Per-column reduction over the 32 lanes of a warp for N = 4, 8 or 16 columns: each of
// the first log2(N) butterfly steps halves the columns a lane carries (it keeps one half
// and trades the other with its partner), the remaining steps combine plain values.
// Afterwards lane l holds the result for column reduce_col<N>(l).  N - 1 + 5 - log2(N)
// shuffles instead of 5 N.
template <int N>
__device__ __forceinline__ int reduce_col(int lane) {
    int col = 0, n = N, m = 16;
#pragma unroll
    for (; n > 1; n >>= 1, m >>= 1)
        if (lane & m) col += n / 2;
    return col;
}

template <int N, bool kMax>
__device__ __forceinline__ float warp_reduce_cols(float (&v)[N], int lane) {
    int m = 16;
#pragma unroll
    for (int n = N; n > 1; n >>= 1, m >>= 1) {
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, m);
            v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
    float r = v[0];
#pragma unroll
    for (; m > 0; m >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, r, m);
        r = kMax ? fmaxf(r, o) : r + o;
    }
    return r;
}

template <bool kBF16>
__device__ __forceinline__ uint16_t to16(float x) {
    uint32_t w = pack2<kBF16>(x, 0.f);
    return (uint16_t)(w & 0xffffu);
}

template <class DC, int GMAX, bool kBF16>
__global__ void __launch_bounds__(kDecThreads, 1)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const DecParams p) {
    constexpr int D = DC::D, DA = DC::DA, SUB = DC::SUB, NS = DC::NS, OM = DC::OM;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t* base_gen = smem_raw + (base - raw_u32);
    // The V ring comes first: an MMA's rows past the data (the second 64-dim atom of V^T at
    // D = 64, the 64 rows past a 64-key K tile at D = 256) then read the next stage, the K
    // ring or the Q buffers, all inside this CTA's shared memory.
    const uint32_t sV = base;
    const uint32_t sK = sV + NS * DC::KVBytes;
    const uint32_t sQ = sK + NS * DC::KVBytes;
    const uint32_t sP = sQ + 2 * DC::QBytes;
    DecSmemTail& T = *reinterpret_cast<DecSmemTail*>(base_gen + DC::TileBytes);
    auto bar = [&](int i) -> uint32_t { return smem_u32(&T.bars[i]); };

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const WaitCtx wc{&T.abort_flag, p.status};

    // ---- setup: barriers, TMEM, and the work-item table from kv_lens
    if (tid == 0) {
        for (int i = 0; i < DC::NumBars; ++i)
            mbar_init(bar(i), (i == DC::BarPFull || i == DC::BarPFull + 1 || i == DC::BarODrained) ? 128u : 1u);
        T.abort_flag = 0;
        T.max_len = 0;
        fence_mbar_init();
    }
    if (warp == kDecMmaWarp) {
        tmem_alloc(smem_u32(&T.tmem_slot), DC::TmemCols);
        tmem_relinquish();
    }
    if (warp == kDecProducerWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    // P^T rows past the group stay zero for the whole kernel.
    for (int i = tid; i < 2 * DC::PBytes / 4; i += kDecThreads)
        reinterpret_cast<uint32_t*>(base_gen + (sP - base))[i] = 0u;
    fence_proxy_async_smem();
    __syncthreads();
    for (int b = tid; b < p.B; b += kDecThreads) {
        const int len = min(max(p.kv_lens[b], 0), p.Smax);
        T.lens[b] = len;
        atomicMax(&T.max_len, len);
    }
    __syncthreads();
    {
        // exclusive scan over b of the tiles of one pair, 128 threads x up to 8 entries each
        const int per_t = (p.B + 127) / 128;
        int local = 0;
        if (tid < 128) {
            for (int i = 0; i < per_t; ++i) {
                const int b = tid * per_t + i;
                if (b < p.B) local += (T.lens[b] + kDecBN - 1) / kDecBN;
            }
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (tid < 128 && lane == 31) T.warp_sums[warp] = incl;
        __syncthreads();
        if (tid < 128) {
            int run = incl - local;
            for (int w = 0; w < warp; ++w) run += T.warp_sums[w];
            for (int i = 0; i < per_t; ++i) {
                const int b = tid * per_t + i;
                if (b < p.B) {
                    T.prefix[b] = run;
                    run += (T.lens[b] + kDecBN - 1) / kDecBN;
                }
            }
            if (tid == 127) T.prefix[p.B] = run;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // This CTA's range of the plan, and its head within a planned group of kv heads.
    const int rng = (int)blockIdx.x / p.kv_group, sub = (int)blockIdx.x % p.kv_group;
    const int Hu = p.Hkv / p.kv_group;
    if (tid == 0) {
        T.total_tiles = Hu * T.prefix[p.B];
        T.width = decode_range_width(T.total_tiles, (T.max_len + kDecBN - 1) / kDecBN,
                                     (int)gridDim.x / p.kv_group, p.ns);
    }
    __syncthreads();
    const uint32_t tmem = T.tmem_slot;
    const int x0 = (int)min((long long)rng * T.width, (long long)T.total_tiles);
    const int x_end = min(x0 + T.width, T.total_tiles);
    // The merge kernel may be scheduled now; it waits for this grid's results itself.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kDecProducerWarp) {
        // -------------------------------------------------------------- producer ----
        if (lane == 0) {
            uint32_t kv_it = 0, icount = 0;
            bool ok = true;
            // Every K/V row is read exactly once by this kernel.
            const uint64_t kv_policy = l2_policy_evict_first();
            int x = x0;
            DecItem it;
            while (ok && next_segment(T, p.B, Hu, rng, p.kv_group, sub, x, x_end, it)) {
                const uint32_t qs = icount & 1u;
                ok = mbar_wait(bar(DC::BarQEmpty + qs), ((icount >> 1) & 1u) ^ 1u, wc);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(DC::BarQFull + qs), DA * p.q_rows * p.sq * 128);
                for (int a = 0; a < DA; ++a)
                    tma_load_4d(sQ + qs * DC::QBytes + a * 2048, &tm_q, bar(DC::BarQFull + qs), a * 64,
                                it.hk * p.group, 0, it.b);
                // Paged caches: a box's page comes from the block table (a page holds a whole
                // number of 128-key tiles, so no box crosses one).  The last step of an item
                // may reach past its tiles (D = 64 steps are 256 keys); such keys are masked,
                // and the table index is clamped so the lookup stays inside the table.
                auto page_of = [&](int r) -> int {
                    return p.block_table[(size_t)it.b * p.max_pages + min(r / p.page_size, p.max_pages - 1)];
                };
                const int nsteps = dec_steps<DC>(it.ntiles);
                for (int j = 0; j < nsteps && ok; ++j) {
                    const uint32_t st = kv_it % NS;
                    const uint32_t ph = ((kv_it / NS) & 1u) ^ 1u;
                    int c2[DC::NBOX], c3[DC::NBOX];
#pragma unroll
                    for (int bx = 0; bx < DC::NBOX; ++bx) {
                        const int row = it.k0 + j * SUB + bx * DC::BOX;
                        c2[bx] = row;      // contiguous: (key row, sequence)
                        c3[bx] = it.b;
                        if (p.block_table) {  // paged: (row within page, page)
                            c2[bx] = row % p.page_size;
                            c3[bx] = page_of(row);
                        }
                    }
                    ok = mbar_wait(bar(DC::BarKEmpty + st), ph, wc);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(DC::BarKFull + st), DC::KVBytes);
                    for (int a = 0; a < DA; ++a)
#pragma unroll
                        for (int bx = 0; bx < DC::NBOX; ++bx)
                            tma_load_4d_hint(sK + st * DC::KVBytes + a * (SUB * 128) + bx * (DC::BOX * 128), &tm_k,
                                             bar(DC::BarKFull + st), a * 64, it.hk, c2[bx], c3[bx], kv_policy);
                    ok = mbar_wait(bar(DC::BarVEmpty + st), ph, wc);
                    if (!ok) {
                        mbar_wait_drain(bar(DC::BarKFull + st), (kv_it / NS) & 1u);
                        break;
                    }
                    mbar_arrive_expect_tx(bar(DC::BarVFull + st), DC::KVBytes);
                    for (int a = 0; a < DA; ++a)
#pragma unroll
                        for (int bx = 0; bx < DC::NBOX; ++bx)
                            tma_load_4d_hint(sV + st * DC::KVBytes + a * (SUB * 128) + bx * (DC::BOX * 128), &tm_v,
                                             bar(DC::BarVFull + st), a * 64, it.hk, c2[bx], c3[bx], kv_policy);
                    ++kv_it;
                }
                ++icount;
            }
            for (uint32_t d = 0; d < (uint32_t)NS && d < kv_it; ++d) {
                const uint32_t last = kv_it - 1 - d;
                mbar_wait_drain(bar(DC::BarKFull + last % NS), (last / NS) & 1u);
                mbar_wait_drain(bar(DC::BarVFull + last % NS), (last / NS) & 1u);
            }
            for (uint32_t d = 0; d < 2u && d < icount; ++d) {
                const uint32_t last = icount - 1 - d;
                mbar_wait_drain(bar(DC::BarQFull + (last & 1u)), (last >> 1) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == kDecMmaWarp) {
        // ------------------------------------------------------------ MMA issuer ----
        // The whole warp runs the issue loop: every lane waits on the barriers and the
        // outcome is voted, and elect.sync picks the lane that issues each MMA and commit.
        // Descriptors are built once; stepping through a tile only moves the start-address
        // field of the low word.  (Uniform control flow keeps each small MMA cheap to issue.)
        {
            constexpr uint32_t idesc_s = make_idesc_f16(128, 16, kBF16, false, false);
            constexpr uint32_t idesc_o = make_idesc_f16(128, 16, kBF16, true, false);
            uint32_t kv_it = 0, icount = 0, it_s = 0;
            bool ok = true;
            auto wait = [&](uint32_t b, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
            };
            const uint64_t dk0 = make_sdesc_sw128(sK, 16, 1024);
            const uint64_t dq0 = make_sdesc_sw128(sQ, 16, 1024);
            const uint64_t dv0 = make_sdesc_sw128(sV, SUB * 128, 1024);
            const uint64_t dp0 = make_sdesc_sw128(sP, 16, 1024);
            const uint32_t k_lo = (uint32_t)dk0, k_hi = (uint32_t)(dk0 >> 32);
            const uint32_t q_lo = (uint32_t)dq0, q_hi = (uint32_t)(dq0 >> 32);
            const uint32_t v_lo = (uint32_t)dv0, v_hi = (uint32_t)(dv0 >> 32);
            const uint32_t p_lo = (uint32_t)dp0, p_hi = (uint32_t)(dp0 >> 32);
            // S^T = K Q^T over the D head dims (16 per MMA), one M block of 128 keys at a time.
            auto issue_s = [&](uint32_t qs, uint32_t kst, uint32_t slot) {
                const uint32_t b = q_lo + ((qs * DC::QBytes) >> 4);
#pragma unroll
                for (int m = 0; m < DC::KM; ++m) {
                    const uint32_t a = k_lo + ((kst * DC::KVBytes + m * (128 * 128)) >> 4);
                    const uint32_t d = tmem + slot * DC::SCols + m * 16;
                    umma_ss_elect<false>(d, a, k_hi, b, q_hi, idesc_s);
#pragma unroll
                    for (int kk = 1; kk < D / 16; ++kk)
                        umma_ss_elect<true>(d, a + (((kk >> 2) * (SUB * 128) + (kk & 3) * 32) >> 4), k_hi,
                                            b + (((kk >> 2) * 2048 + (kk & 3) * 32) >> 4), q_hi, idesc_s);
                }
            };
            // O^T += V^T P^T over the SUB keys of the tile, one 128-row block of head dims
            // (two 64-dim atoms of the V tile) at a time.
            auto issue_pv = [&](uint32_t vst, uint32_t pbuf, bool acc) {
                const uint32_t b = p_lo + ((pbuf * DC::PBytes) >> 4);
#pragma unroll
                for (int ob = 0; ob < OM; ++ob) {
                    const uint32_t a = v_lo + ((vst * DC::KVBytes + ob * 2 * (SUB * 128)) >> 4);
                    const uint32_t d = tmem + DC::OCol0 + ob * 16;
                    if (acc)
                        umma_ss_elect<true>(d, a, v_hi, b, p_hi, idesc_o);
                    else
                        umma_ss_elect<false>(d, a, v_hi, b, p_hi, idesc_o);
#pragma unroll
                    for (int kk = 1; kk < SUB / 16; ++kk)
                        umma_ss_elect<true>(d, a + ((kk * (16 * 128)) >> 4), v_hi,
                                            b + (((kk >> 2) * 2048 + (kk & 3) * 32) >> 4), p_hi, idesc_o);
                }
            };
            int x = x0;
            DecItem item;
            while (ok && next_segment(T, p.B, Hu, rng, p.kv_group, sub, x, x_end, item)) {
                const int n = dec_steps<DC>(item.ntiles);  // MMA steps of this item
                const uint32_t qs = icount & 1u;
                ok = wait(bar(DC::BarQFull + qs), (icount >> 1) & 1u);
                if (!ok) break;
                {
                    const uint32_t st = kv_it % NS;
                    ok = wait(bar(DC::BarKFull + st), (kv_it / NS) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(qs, st, it_s & 1u);
                    umma_commit_elect(bar(DC::BarSFull + (it_s & 1u)));
                    umma_commit_elect(bar(DC::BarKEmpty + st));
                    if (n == 1) umma_commit_elect(bar(DC::BarQEmpty + qs));
                }
                for (int j = 0; j < n && ok; ++j) {
                    const uint32_t cur = kv_it + j;
                    const uint32_t st = cur % NS;
                    if (j + 1 < n) {
                        const uint32_t nst = (cur + 1) % NS;
                        ok = wait(bar(DC::BarKFull + nst), ((cur + 1) / NS) & 1u);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(qs, nst, (it_s + 1) & 1u);
                        umma_commit_elect(bar(DC::BarSFull + ((it_s + 1) & 1u)));
                        umma_commit_elect(bar(DC::BarKEmpty + nst));
                        if (j + 2 == n) umma_commit_elect(bar(DC::BarQEmpty + qs));
                    }
                    ok = wait(bar(DC::BarPFull + (it_s & 1u)), (it_s >> 1) & 1u);
                    if (ok && j == 0 && icount > 0) ok = wait(bar(DC::BarODrained), (icount - 1) & 1u);
                    if (ok) ok = wait(bar(DC::BarVFull + st), (cur / NS) & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(st, it_s & 1u, j > 0);
                    umma_commit_elect(bar(DC::BarODone + (it_s & 1u)));
                    umma_commit_elect(bar(DC::BarVEmpty + st));
                    ++it_s;
                }
                kv_it += n;
                ++icount;
            }
            // Every MMA issued has completed before TMEM and shared memory are released.
            umma_commit_elect(bar(DC::BarFinal));
            mbar_wait_drain(bar(DC::BarFinal), 0);
            __syncwarp();
        }
    } else {
        // --------------------------------------------------------- compute warps ----
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const float kNegInf = -__int_as_float(0x7f800000);
        const int g = p.group;
        uint32_t it_s = 0;
        bool ok = true;
        int x = x0;
        DecItem item;
        while (ok && next_segment(T, p.B, Hu, rng, p.kv_group, sub, x, x_end, item)) {
            float m_run[GMAX], l_part[GMAX];
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                m_run[h] = kNegInf;
                l_part[h] = 0.f;
            }
            const int n = dec_steps<DC>(item.ntiles);
            for (int j = 0; j < n; ++j) {
                const uint32_t slot = it_s & 1u;
                ok = mbar_wait(bar(DC::BarSFull + slot), (it_s >> 1) & 1u, wc);
                if (!ok) break;
                tc_fence_after();
                // TMEM lane tid of S^T block m holds key k0 + j SUB + 128 m + tid; lanes past
                // SUB (64-key steps) hold no key.
                uint32_t u[DC::KM][16];
#pragma unroll
                for (int m = 0; m < DC::KM; ++m) tmem_ld_32x32b_x16(lane_base + slot * DC::SCols + m * 16, u[m]);
#pragma unroll
                for (int m = 0; m < DC::KM; ++m) tmem_wait_ld(u[m]);
                const int ncols = g * p.sq;
                // Token s sees keys <= len - sq + s; column h holds token h / g, so with
                // causal tokens a key is visible to columns h >= (key - len + sq) * g.
                const int lim0 = T.lens[item.b] - p.sq;
                float sv[DC::KM][GMAX], mx[GMAX];
#pragma unroll
                for (int h = 0; h < GMAX; ++h) mx[h] = kNegInf;
#pragma unroll
                for (int m = 0; m < DC::KM; ++m) {
                    const int kin = m * 128 + tid;  // key within the step
                    const int key = item.k0 + j * SUB + kin;
                    const int h_lo = p.causal ? max(key - lim0, 0) * g : 0;
                    const int h_hi = (kin < SUB && key < item.k1) ? ncols : 0;  // columns [h_lo, h_hi)
#pragma unroll
                    for (int h = 0; h < GMAX; ++h) {
                        const bool vis = h >= h_lo && h < h_hi;
                        sv[m][h] = vis ? __uint_as_float(u[m][h]) : kNegInf;
                        mx[h] = fmaxf(mx[h], sv[m][h]);
                    }
                }
                // per-column max over this warp's 32 keys, then over the four warps
                const float wm = warp_reduce_cols<GMAX, true>(mx, lane);
                if ((lane & (32 / GMAX - 1)) == 0) T.red[j & 1][warp][reduce_col<GMAX>(lane)] = wm;
                named_bar_sync(1, 128);
                float mb4[GMAX];
#pragma unroll
                for (int h4 = 0; h4 < GMAX; h4 += 4) {
                    float4 r[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) r[w] = *reinterpret_cast<const float4*>(&T.red[j & 1][w][h4]);
                    mb4[h4 + 0] = fmaxf(fmaxf(r[0].x, r[1].x), fmaxf(r[2].x, r[3].x));
                    mb4[h4 + 1] = fmaxf(fmaxf(r[0].y, r[1].y), fmaxf(r[2].y, r[3].y));
                    mb4[h4 + 2] = fmaxf(fmaxf(r[0].z, r[1].z), fmaxf(r[2].z, r[3].z));
                    mb4[h4 + 3] = fmaxf(fmaxf(r[0].w, r[1].w), fmaxf(r[2].w, r[3].w));
                }
                float alpha[GMAX], msub[GMAX];
                bool any_rescale = false;
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    const float mb = mb4[h] * p.scale_log2;
                    const bool bump = mb > m_run[h] + 8.0f;
                    const float mn = bump ? mb : m_run[h];
                    alpha[h] = bump ? ex2_approx(m_run[h] - mn) : 1.0f;
                    any_rescale |= bump;
                    m_run[h] = mn;
                    msub[h] = (mn == kNegInf) ? 0.f : mn;
                }
                float pv[DC::KM][GMAX];
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    float ps = 0.f;
#pragma unroll
                    for (int m = 0; m < DC::KM; ++m) {
                        pv[m][h] = ex2_approx(fmaf(sv[m][h], p.scale_log2, -msub[h]));
                        ps += pv[m][h];
                    }
                    l_part[h] = l_part[h] * alpha[h] + ps;
                }
                // This tile's P^T buffer was last read by the P.V of tile it_s - 2.
                if (it_s >= 2) {
                    ok = mbar_wait(bar(DC::BarODone + (it_s & 1u)), ((it_s - 2) >> 1) & 1u, wc);
                    if (!ok) break;
                }
                if (j > 0 && any_rescale) {  // uniform: every thread saw the same maxima
                    // the previous P.V must have finished accumulating into O
                    ok = mbar_wait(bar(DC::BarODone + ((it_s - 1) & 1u)), ((it_s - 1) >> 1) & 1u, wc);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int ob = 0; ob < OM; ++ob) {
                        uint32_t ov[16];
                        tmem_ld_32x32b_x16(lane_base + DC::OCol0 + ob * 16, ov);
                        tmem_wait_ld(ov);
#pragma unroll
                        for (int h = 0; h < GMAX; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
                        tmem_st_32x32b_x16(lane_base + DC::OCol0 + ob * 16, ov);
                    }
                    tmem_wait_st();
                }
                const uint32_t sPb = sP + (it_s & 1u) * DC::PBytes;
#pragma unroll
                for (int m = 0; m < DC::KM; ++m) {
                    const int kin = m * 128 + tid;
                    if (kin < SUB) {
#pragma unroll
                        for (int h = 0; h < GMAX; ++h) st_shared_u16(pt_addr(sPb, h, kin), to16<kBF16>(pv[m][h]));
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(DC::BarPFull + (it_s & 1u)));
                ++it_s;
            }
            if (!ok) break;
            // ---- end of item: O^T / l -> partial output, log-sum-exp per head
            ok = mbar_wait(bar(DC::BarODone + ((it_s - 1) & 1u)), ((it_s - 1) >> 1) & 1u, wc);
            if (!ok) break;
            tc_fence_after();
            uint32_t ov[OM][16];
#pragma unroll
            for (int ob = 0; ob < OM; ++ob) tmem_ld_32x32b_x16(lane_base + DC::OCol0 + ob * 16, ov[ob]);
            tmem_wait_ld(ov[0]);
#pragma unroll
            for (int ob = 1; ob < OM; ++ob) tmem_wait_ld(ov[ob]);
            tc_fence_before();
            mbar_arrive(bar(DC::BarODrained));
            {
                float ls[GMAX];
#pragma unroll
                for (int h = 0; h < GMAX; ++h) ls[h] = l_part[h];
                const float wl = warp_reduce_cols<GMAX, false>(ls, lane);
                if ((lane & (32 / GMAX - 1)) == 0) T.lred[warp][reduce_col<GMAX>(lane)] = wl;
            }
            named_bar_sync(1, 128);
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                const float lt = (T.lred[0][h] + T.lred[1][h]) + (T.lred[2][h] + T.lred[3][h]);
                if (h < g * p.sq) {
                    // column h is (token h / g, head hk * g + h % g); rows are [B, sq, Hq]
                    const size_t qrow = ((size_t)item.b * p.sq + h / g) * p.Hq + (size_t)item.hk * g + h % g;
                    const size_t row = qrow * p.ns + item.c;
                    // thread tid owns head dim tid of every 128-row block of O^T
#pragma unroll
                    for (int ob = 0; ob < OM; ++ob) {
                        const int dim = ob * 128 + tid;
                        if (dim < D) p.o_part[row * D + dim] = lt > 0.f ? __uint_as_float(ov[ob][h]) / lt : 0.f;
                    }
                    if (tid == 0)
                        p.lse_part[row] =
                            lt > 0.f ? (m_run[h] + lg2_approx(lt)) * 0.69314718055994531f : kNegInf;
                }
            }
            // lred is rewritten only after the next item's per-tile barriers
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kDecMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, DC::TmemCols);
    }
}

// Merge kernel: one warp per (b, query head); lane l owns head dims l, l + 32, ...
template <int D, bool kBF16>
__global__ void __launch_bounds__(128)
    fa_decode_combine_kernel(const DecParams p) {
    constexpr int V = D / 32;  // head dims per lane
    // The split kernel's range width, from the same lengths.
    __shared__ int s_max_len, s_sum_tiles;
    if (threadIdx.x == 0) {
        s_max_len = 0;
        s_sum_tiles = 0;
    }
    __syncthreads();
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
        const int len = min(max(p.kv_lens[b], 0), p.Smax);
        atomicMax(&s_max_len, len);
        atomicAdd(&s_sum_tiles, (len + kDecBN - 1) / kDecBN);
    }
    __syncthreads();
    const int Hu = p.Hkv / p.kv_group;
    const int W = decode_range_width(Hu * s_sum_tiles, (s_max_len + kDecBN - 1) / kDecBN,
                                     p.split_grid / p.kv_group, p.ns);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x * 4 + warp;  // row of [B, sq, Hq]
    if (bh >= p.B * p.sq * p.Hq) return;
    const int b = bh / (p.sq * p.Hq);
    const int s_tok = (bh / p.Hq) % p.sq;
    const int hq = bh % p.Hq;
    const int len = min(max(p.kv_lens[b], 0), p.Smax);
    // This row's pair (b, kv head) starts after the tiles of all earlier plan entries; it
    // has one partial per range it meets.
    int before = 0;  // tiles of one pair of each sequence before b
    for (int bb = lane; bb < b; bb += 32) before += (min(max(p.kv_lens[bb], 0), p.Smax) + kDecBN - 1) / kDecBN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    const int tb = (len + kDecBN - 1) / kDecBN;
    const int pstart = Hu * before + (hq / p.group / p.kv_group) * tb;
    const int n = tb > 0 ? (pstart + tb - 1) / W - pstart / W + 1 : 0;
    const float kNegInf = -__int_as_float(0x7f800000);
    const float kLog2e = 1.4426950408889634f;
    const float* lrow = p.lse_part + (size_t)bh * p.ns;
    const float* orow = p.o_part + (size_t)bh * p.ns * D + lane;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    float lse = kNegInf;
    // The partials are written by the split kernel, which may still be running when this
    // grid starts (programmatic dependent launch): wait for its completion here.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Up to NB pieces (all of them at the decode workload's sizes): every piece's LSE and
    // partial output are loaded together, one round trip to memory after the wait, and
    // each lane combines them in piece order.  More pieces: the maximum first, then
    // batches of NB.  Slots past n reload piece n - 1 with weight 0, an exact zero.
    constexpr int NB = V <= 4 ? 16 : 8;
    if (n > 0 && n <= NB) {
        float l[NB], v[NB][V];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int cu = min(u, n - 1);
            l[u] = lrow[cu];
#pragma unroll
            for (int i = 0; i < V; ++i) v[u][i] = orow[(size_t)cu * D + i * 32];
        }
        float m = kNegInf;
#pragma unroll
        for (int u = 0; u < NB; ++u) m = fmaxf(m, l[u]);
        // m = -inf: no piece holds a visible key for this row (a causal token that sees
        // none): O = 0, LSE = -inf.
        if (m != kNegInf) {
            float s = 0.f;
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const float w = u < n ? ex2_approx((l[u] - m) * kLog2e) : 0.f;
                s += w;
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] = fmaf(w, v[u][i], acc[i]);
            }
            const float inv = 1.0f / s;
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] *= inv;
            lse = m + lg2_approx(s) * 0.69314718055994531f;
        }
    } else if (n > NB) {
        float m = kNegInf;
        for (int c = lane; c < n; c += 32) m = fmaxf(m, lrow[c]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (m != kNegInf) {
            float s = 0.f;
            for (int c = 0; c < n; c += NB) {
                float v[NB][V];
                float w[NB];
#pragma unroll
                for (int u = 0; u < NB; ++u) {
                    const int cu = min(c + u, n - 1);
#pragma unroll
                    for (int i = 0; i < V; ++i) v[u][i] = orow[(size_t)cu * D + i * 32];
                    w[u] = c + u < n ? ex2_approx((lrow[cu] - m) * kLog2e) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < NB; ++u) {
                    s += w[u];
#pragma unroll
                    for (int i = 0; i < V; ++i) acc[i] = fmaf(w[u], v[u][i], acc[i]);
                }
            }
            const float inv = 1.0f / s;
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] *= inv;
            lse = m + lg2_approx(s) * 0.69314718055994531f;
        }
    }
    uint16_t* out = reinterpret_cast<uint16_t*>(p.o) + (size_t)bh * D + lane;
#pragma unroll
    for (int i = 0; i < V; ++i) out[i * 32] = to16<kBF16>(acc[i]);
    if (p.lse && lane == 0) p.lse[((size_t)b * p.Hq + hq) * p.sq + s_tok] = lse;
}

template <class DC, int GMAX, bool kBF16>
static fa_status launch_split(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecParams& p, int grid, cudaStream_t s) {
    static int attr[64] = {0};
    auto kern = fa_decode_split_kernel<DC, GMAX, kBF16>;
    if (!ensure_smem_attr((const void*)kern, DC::SmemBytes, attr)) return FA_ERR_CUDA;
    kern<<<grid, kDecThreads, DC::SmemBytes, s>>>(tq, tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Host launcher for head dim D: tensor maps, parameters, the split kernel and the merge.
template <int D>
fa_status launch_decode_d(const DecodeArgs& a, cudaStream_t s) {
    using DC = DecCfg<D>;
    if (a.D != D) return FA_ERR_UNSUPPORTED;
    if (a.B > kDecMaxB) return FA_ERR_UNSUPPORTED;
    const int g = a.Hq / a.Hkv;
    CUtensorMap tq, tk, tv;
    const int g_cols = (a.Hq / a.Hkv) * a.sq;  // MMA N columns in use
    if (g_cols > 16) return FA_ERR_UNSUPPORTED;
    const int q_rows = a.sq == 1 ? (a.Hq < 16 ? a.Hq : 16) : a.Hq / a.Hkv;
    // Contiguous caches are [B, Smax, Hkv, D]; paged pools are [num_pages, page_size, Hkv, D].
    const uint64_t rows_dim = a.block_table ? (uint64_t)a.page_size : (uint64_t)a.Smax;
    const uint64_t outer_dim = a.block_table ? (uint64_t)a.num_pages : (uint64_t)a.B;
    if (!encode_tmap_4d_box(&tq, a.q, a.bf16, a.D, a.Hq, a.sq, a.B, q_rows, a.sq) ||
        !encode_tmap_4d(&tk, a.k_cache, a.bf16, a.D, a.Hkv, rows_dim, outer_dim, DC::BOX) ||
        !encode_tmap_4d(&tv, a.v_cache, a.bf16, a.D, a.Hkv, rows_dim, outer_dim, DC::BOX))
        return FA_ERR_CUDA;
    DecParams p;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.group = g;
    p.Smax = a.Smax;
    p.ns = a.num_splits;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.kv_lens = a.kv_lens;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    p.o = a.o;
    p.lse = a.lse;
    p.status = a.dev_status;
    p.q_rows = q_rows;
    p.sq = a.sq;
    p.causal = a.causal ? 1 : 0;
    p.block_table = a.block_table;
    p.page_size = a.page_size;
    p.max_pages = a.max_pages;
    // One CTA per SM; the kernel cuts the work into equal ranges of tiles, one per group of
    // g CTAs, g the largest of 8, 4 and 2 that divides Hkv (and is at most the SM count),
    // else 1.  The grid is the largest multiple of g up to the SM count.
    int kvg = 1;
    for (int c = kDecMaxKvGroup; c >= 2; c >>= 1)
        if (a.Hkv % c == 0 && a.num_sms >= c) {
            kvg = c;
            break;
        }
    p.kv_group = kvg;
    const int grid = a.num_sms - a.num_sms % kvg;
    p.split_grid = grid;
    fa_status st;
    if (g_cols <= 4)
        st = a.bf16 ? launch_split<DC, 4, true>(tq, tk, tv, p, grid, s)
                    : launch_split<DC, 4, false>(tq, tk, tv, p, grid, s);
    else if (g_cols <= 8)
        st = a.bf16 ? launch_split<DC, 8, true>(tq, tk, tv, p, grid, s)
                    : launch_split<DC, 8, false>(tq, tk, tv, p, grid, s);
    else
        st = a.bf16 ? launch_split<DC, 16, true>(tq, tk, tv, p, grid, s)
                    : launch_split<DC, 16, false>(tq, tk, tv, p, grid, s);
    if (st != FA_OK) return st;
    // The merge kernel is launched as a programmatic dependent of the split kernel: its
    // launch overlaps the split kernel's tail, and it waits for the split results itself.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.B * a.sq * a.Hq + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = a.bf16 ? cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D, true>, p)
                                 : cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D, false>, p);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
