// fa_fwd.cuh -- exact attention forward for sm_103a (tcgen05 + TMA, warp-specialised).
//
// What is computed: O = softmax(scale * Q K^T [+ causal mask]) V with the per-row
// log-sum-exp, for [B, S, H, D] tensors with grouped-query heads (page
// "flash-attention-v100", "How to use FlashAttention"; bottom-right causal mask from
// "Changelog", "2.1: Change behavior of causal flag").
//
// How (FlashAttention-2 work partitioning, page "ampere_flash_attention_from_scratch";
// the RTX 3080 kernel there is prior art, this is a Blackwell design):
//  * A persistent CTA per SM walks work tiles (b, h, query block of NQ x 128 rows); the
//    query blocks of one head are adjacent in the walk so concurrent CTAs share K/V in L2.
//    In causal batches a CTA takes query blocks qb and nqb - 1 - qb of a head back to
//    back: their key ranges add up to the same length, so the CTAs get even work.
//  * Warp roles: one TMA producer warp streams Q once per tile and K/V tiles of BN keys
//    through an NS-stage ring (full / empty mbarriers); one MMA warp issues tcgen05.mma
//    (the whole warp runs the issue loop, elect.sync picks the issuing lane); NQ softmax
//    warpgroups own one 128-row Q tile each (thread = row = TMEM lane).
//  * S = Q K^T: A = Q and B = K from 128-byte-swizzled shared memory, fp32 accumulator in
//    TMEM.  The softmax warpgroup reads S from TMEM, applies the mask, keeps the running
//    max m and sum l (online softmax in base 2 with scale*log2(e) folded into one FMA),
//    rounds P to 16 bits and writes it back into the same TMEM columns.
//  * O += P V: A = P straight from TMEM, B = V (MN-major) from shared memory.  O stays in
//    TMEM for the whole KV loop; it is rescaled only when a row max grows by more than
//    2^8 (the sum l uses the same stale max, so the final O / l is exact).
//  * With NQ = 2 the two Q tiles ping-pong: the tensor pipe runs one tile's GEMMs while
//    the other tile's softmax runs.  With NQ = 1 S is double-buffered instead.  At D = 64,
//    where S, P and O of both tiles fit in TMEM side by side, P has columns of its own and
//    the next S of a tile is issued as soon as the softmax has read the current one.
//  * Sliding windows (fixed-length batches) use an instantiation that skips, per Q tile,
//    the blocks outside that tile's window.
//  * Epilogue: O / l rounded to 16 bits, staged in shared memory in the TMA layout and
//    written by a store warp with TMA stores (row stores for packed variable-length
//    batches); LSE = (m + log2 l) ln 2.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

struct FwdParams {
    int B, Sq, Sk, Hq, Hkv, group;
    int causal;
    // Sliding window (page "flash-attention-v100", flash_attn_func window_size): query i
    // sees keys in [i + Sk - Sq - win_left, i + Sk - Sq + hi_off]; has_lo / has_hi say
    // whether each bound applies (hi_off = 0 under the causal flag).
    int has_lo, win_left, has_hi, hi_off;
    float scale_log2;  // softmax scale * log2(e)
    int num_qb;        // query blocks of NQ * 128 rows per (b, h) (fixed-length batches)
    int num_tiles;     // tile indices the CTAs walk (fixed-length batches)
    // Causal batches: query blocks qb and nqb - 1 - qb of a (sequence, head), whose key
    // ranges add up to the same length for every qb, go to the same CTA one after the
    // other, so CTAs get even work.  Tile index t = (2 v + m) * grid + c names pair
    // v * grid + c, member m (0: the long block, 1: the short one).
    int pair_tiles;
    // Variable-length batches (page "flash-attention-v100", "Changelog", "2.0",
    // flash_attn_varlen_func): sequence b holds query rows [cu_q[b], cu_q[b+1]) of a packed
    // [total_q, Hq, D] tensor and key rows [cu_k[b], cu_k[b+1]) of [total_k, Hkv, D];
    // null for fixed-length [B, S, H, D] batches.  LSE is then [Hq, total_q].
    const int32_t* cu_q;
    const int32_t* cu_k;
    int total_q;
    void* o;           // [B, Sq, Hq, D]
    float* lse;        // [B, Hq, Sq] or null
    int* status;       // sticky device status word
};

constexpr int kMaxVarlenB = 1024;

// Work-tile table of a variable-length batch, built by every CTA at start.
struct VarlenTable {
    // Sequences are walked longest first: order[k] is the k-th longest (by query blocks,
    // ties by index), and prefix[k] is the exclusive prefix of Hq * ceil(Sq / (NQ * 128))
    // (of pairs of blocks, when paired) over that order.  CTAs that run together then
    // work on blocks of the same length and stay in step, sharing K/V in L2, and the
    // short sequences fill in at the end.
    int order[kMaxVarlenB];
    int prefix[kMaxVarlenB + 1];
    int q0[kMaxVarlenB + 1];      // cu_seqlens_q
    int k0[kMaxVarlenB + 1];      // cu_seqlens_k
};

template <int D_, int BN_, int NQ_, int NS_>
struct FwdConfig {
    static constexpr int D = D_;
    static constexpr int BM = 128;
    static constexpr int BN = BN_;
    static constexpr int NQ = NQ_;
    static constexpr int NS = NS_;
    static constexpr int DA = (D + 63) / 64;  // 128-byte column atoms per row
    static constexpr int kQBytes = BM * DA * 128;
    static constexpr int kKVBytes = BN * DA * 128;
    static constexpr int kSlots = (NQ == 1) ? 2 : NQ;  // S buffers in TMEM
    // S ahead of P.V with two Q tiles: where S, P and O of both tiles fit in TMEM side by
    // side (D = 64), P gets BN / 2 columns of its own instead of overwriting S.  The
    // softmax then hands S back as soon as it has read it into registers, and the next
    // S = Q K^T of the same tile runs while this block's exponentials are computed; the
    // chain S -> softmax -> P.V -> S of one tile no longer paces the loop.
    static constexpr bool kSAhead = (NQ == 2) && (NQ * BN + NQ * (BN / 2) + NQ * D <= 512);
    static constexpr int kPCol0 = NQ * BN;  // first P column (kSAhead)
    static constexpr int kOCol0 = kSAhead ? NQ * BN + NQ * (BN / 2) : kSlots * BN;  // first O column
    static constexpr int kTmemCols = 512;
    static_assert(kOCol0 + NQ * D <= kTmemCols, "TMEM budget");
    static_assert(D % 32 == 0 && BN % 32 == 0, "tile shape");
    static constexpr int kThreads = 128 * NQ + 96;
    // O-done is signalled after every P.V when S is issued ahead of P.V (NQ == 1, or
    // kSAhead), and only after a tile's last P.V otherwise.
    static constexpr bool kOPerIter = (NQ == 1) || kSAhead;
    // With two Q tiles the K/V ring stages are released by the second softmax warpgroup.
    // S1(j) completing implies S0(j) and every P.V issued before S1(j) completed, so K_j
    // is free, and so is V_{j-1} (P.V of block j - 1 precedes S(j) in the issue order), or
    // V_{j-2} with kSAhead (S(j) is issued ahead of P.V of block j - 1).  That saves the
    // tensor pipe two tcgen05.commit per iteration.
    static constexpr bool kRingBySoftmax = (NQ > 1);
    static constexpr uint32_t kVReleaseLag = kSAhead ? 2u : 1u;
    static constexpr int kProducerWarp = 4 * NQ;
    static constexpr int kMmaWarp = 4 * NQ + 1;
    // O is written through shared memory: a softmax warpgroup stages its normalised tile
    // there in the TMA layout and this warp stores it with TMA bulk stores, so the softmax
    // warps do not issue row-strided global stores.  The staging buffer holds one or two
    // 64-column atoms (see Layout); wider tiles are staged in rounds.
    static constexpr int kStoreWarp = 4 * NQ + 2;
    // barrier indices
    static constexpr int kBarQFull = 0;
    static constexpr int kBarQEmpty = kBarQFull + NQ;
    static constexpr int kBarKFull = kBarQEmpty + NQ;
    static constexpr int kBarKEmpty = kBarKFull + NS;
    static constexpr int kBarVFull = kBarKEmpty + NS;
    static constexpr int kBarVEmpty = kBarVFull + NS;
    static constexpr int kBarSFull = kBarVEmpty + NS;
    static constexpr int kBarPFull = kBarSFull + kSlots;
    static constexpr int kBarODone = kBarPFull + NQ;
    static constexpr int kBarODrained = kBarODone + NQ;
    static constexpr int kBarFinal = kBarODrained + NQ;
    static constexpr int kBarStaged = kBarFinal + 1;     // a warpgroup staged one round of O
    static constexpr int kBarStageFree = kBarStaged + 1;  // per Q tile: the buffer is yours
    static constexpr int kBarSFree = kBarStageFree + NQ;  // per Q tile: S read (kSAhead)
    static constexpr int kNumBars = kBarSFree + NQ;
    // Shared memory of one instantiation.  Packed variable-length batches store O row by
    // row and hold their tile table instead of a staging buffer (a 128-row box could reach
    // into the next sequence, and a one-atom buffer staged in rounds measured slower than
    // the row stores).
    template <bool kVarlen>
    struct Layout {
        static constexpr int kStageAtoms = DA < 2 ? DA : 2;
        static constexpr int kStageRounds = DA / kStageAtoms;
        static_assert(DA % kStageAtoms == 0, "staging rounds");
        static constexpr int kStage = kVarlen ? 0 : kStageAtoms * BM * 128;
        static constexpr int kTileBytes = NQ * kQBytes + 2 * NS * kKVBytes + kStage;
        static constexpr int kSmemBytes = 1024 /* alignment slack */ + kTileBytes + 8 * kNumBars + 16 +
                                          (kVarlen ? (int)sizeof(VarlenTable) : 0);
        static_assert(kSmemBytes <= 232448, "shared memory budget");
    };
};

struct TileCoord {
    int b, h, hk, m0, j0, n_kv;  // K/V blocks j0 .. j0 + n_kv - 1; n_kv < 0: no such tile
    int sq, sk;                  // this sequence's query and key lengths
    int q_base, k_base, tb;      // TMA row offsets and outer coordinate of the sequence
    long long o_row0;            // packed output row of query 0 of this sequence
    long long lse0;              // LSE index of (this sequence, this head, query 0)
};

template <class C>
__device__ __forceinline__ TileCoord decode_tile(const FwdParams& p, const VarlenTable* vt, int t) {
    TileCoord c;
    int qb_raw, bh_local, nqb;
    if (vt) {
        // With pairing the prefix counts pairs of query blocks (see pair_tiles).
        int u = t, w = 0;
        if (p.pair_tiles) {
            const int g = (int)gridDim.x;
            w = t / g;
            u = (w >> 1) * g + (t - w * g);
            if (u >= vt->prefix[p.B]) {
                c.n_kv = -1;
                return c;
            }
        }
        int lo = 0, hi = p.B;  // largest k with prefix[k] <= u
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (vt->prefix[mid] <= u) lo = mid; else hi = mid;
        }
        const int local = u - vt->prefix[lo];
        lo = vt->order[lo];  // the sequence
        c.b = lo;
        c.sq = vt->q0[lo + 1] - vt->q0[lo];
        c.sk = vt->k0[lo + 1] - vt->k0[lo];
        nqb = (c.sq + C::NQ * C::BM - 1) / (C::NQ * C::BM);
        if (p.pair_tiles) {
            const int pairs = (nqb + 1) >> 1;
            bh_local = local / pairs;
            const int k = local - bh_local * pairs;
            qb_raw = (w & 1) ? nqb - 1 - k : k;
            if ((w & 1) && nqb - 1 - k == k) {
                c.n_kv = -1;
                return c;
            }
        } else {
            qb_raw = local % nqb;
            bh_local = local / nqb;
        }
        c.h = bh_local;
        c.q_base = vt->q0[lo];
        c.k_base = vt->k0[lo];
        c.tb = 0;
        c.o_row0 = vt->q0[lo];
        c.lse0 = (long long)c.h * p.total_q + vt->q0[lo];
    } else {
        nqb = p.num_qb;
        int bh;
        if (p.pair_tiles) {
            const int g = (int)gridDim.x;
            const int w = t / g;
            const int pairs = (nqb + 1) >> 1;
            const int v = (w >> 1) * g + (t - w * g);
            bh = v / pairs;
            const int k = v - bh * pairs;
            // qb_raw counts from the longest block; member 1 of the middle block of an odd
            // count, and pairs past the last head, are not tiles.
            qb_raw = (w & 1) ? nqb - 1 - k : k;
            if (bh >= p.B * p.Hq || ((w & 1) && nqb - 1 - k == k)) {
                c.n_kv = -1;
                return c;
            }
        } else {
            qb_raw = t % nqb;
            bh = t / nqb;
        }
        c.h = bh % p.Hq;
        c.b = bh / p.Hq;
        c.sq = p.Sq;
        c.sk = p.Sk;
        c.q_base = 0;
        c.k_base = 0;
        c.tb = c.b;
        c.o_row0 = (long long)c.b * p.Sq;
        c.lse0 = ((long long)c.b * p.Hq + c.h) * p.Sq;
    }
    // causal: the longest query block of each head first
    const int qb = p.causal ? (nqb - 1 - qb_raw) : qb_raw;
    c.hk = c.h / p.group;
    c.m0 = qb * (C::NQ * C::BM);
    const int off = c.sk - c.sq;
    const int last_row = min(c.sq, c.m0 + C::NQ * C::BM) - 1;
    long long kv_end = c.sk, kv_begin = 0;
    if (p.has_hi) kv_end = min(kv_end, (long long)last_row + off + p.hi_off + 1);
    if (p.has_lo) kv_begin = max(kv_begin, (long long)c.m0 + off - p.win_left);
    if (kv_end > kv_begin) {
        c.j0 = (int)(kv_begin / C::BN);
        c.n_kv = (int)((kv_end + C::BN - 1) / C::BN) - c.j0;
    } else {
        c.j0 = 0;
        c.n_kv = 0;
    }
    return c;
}

// Blocks [lo, hi] of tile c (indices into its n_kv blocks) that hold a key visible to some
// row of Q sub-tile q; the others are fully masked for that sub-tile and are skipped (no S,
// no softmax, no P.V for it).  With two Q tiles the tile's block range is the union of
// both sub-tiles' ranges, so under a causal mask or a window each sub-tile can have blocks
// of the other's only.  lo > hi: no visible key (rows past the sequence, or rows that see
// no key).  Single-tile and S-ahead configurations always take the whole range.  Only the
// kernel instantiated for sliding windows skips (kSkip): there a tile's first and last
// blocks are each outside one sub-tile's window.  Elsewhere the skipping code cost more
// than it saved, so the other instantiations keep the plain loop.
template <class C>
__device__ __forceinline__ void sub_tile_blocks(const FwdParams& p, const TileCoord& c, int q, int& lo, int& hi) {
    lo = 0;
    hi = c.n_kv - 1;
    if (C::NQ == 1 || C::kSAhead) return;
    const int r0 = c.m0 + q * C::BM;
    const int r1 = min(r0 + C::BM, c.sq) - 1;  // last row of the sub-tile inside the sequence
    const int off = c.sk - c.sq;
    long long kmax = (long long)c.sk - 1, kmin = 0;
    if (p.has_hi) kmax = min(kmax, (long long)r1 + off + p.hi_off);
    if (p.has_lo) kmin = max(kmin, (long long)r0 + off - p.win_left);
    if (r0 >= c.sq || kmax < kmin) {
        lo = 0;
        hi = -1;
        return;
    }
    lo = max(lo, (int)(kmin / C::BN) - c.j0);
    hi = min(hi, (int)(kmax / C::BN) - c.j0);
}

template <class C, bool kBF16, bool kVarlen, bool kSkip = false>
__global__ void __launch_bounds__(C::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
    using L = typename C::template Layout<kVarlen>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t* base_gen = smem_raw + (base - raw_u32);

    const uint32_t sQ = base;
    const uint32_t sK = sQ + C::NQ * C::kQBytes;
    const uint32_t sV = sK + C::NS * C::kKVBytes;
    const uint32_t sStage = sV + C::NS * C::kKVBytes;  // O staging (fixed-length batches)
    const uint32_t sBar = sStage + L::kStage;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_gen + L::kTileBytes + 8 * C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    VarlenTable* vtab = kVarlen ? reinterpret_cast<VarlenTable*>(tmem_slot + 4) : nullptr;

    auto bar = [&](int i) -> uint32_t { return sBar + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WaitCtx wc{abort_flag, p.status};
    constexpr bool kOPerIter = C::kOPerIter;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNumBars; ++i) {
            const bool by_warpgroup = (i >= C::kBarPFull && i < C::kBarPFull + C::NQ) ||
                                      (i >= C::kBarODrained && i < C::kBarODrained + C::NQ) ||
                                      (i >= C::kBarSFree && i < C::kBarSFree + C::NQ) ||
                                      i == C::kBarStaged;
            mbar_init(bar(i), by_warpgroup ? 4u : 1u);  // one elected arrive per warp
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == C::kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == C::kProducerWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_o);
    }
    int num_tiles = p.num_tiles;
    if (vtab) {
        for (int i = threadIdx.x; i <= p.B; i += blockDim.x) {
            vtab->q0[i] = p.cu_q[i];
            vtab->k0[i] = p.cu_k[i];
        }
        __syncthreads();
        auto qblocks = [&](int b) -> int {
            const int sq = max(vtab->q0[b + 1] - vtab->q0[b], 0);
            return (sq + C::NQ * C::BM - 1) / (C::NQ * C::BM);
        };
        // Rank of each sequence by query blocks (descending, ties by index): B <= 1024, so
        // at most B^2 / blockDim comparisons per thread.
        for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
            const int ni = qblocks(i);
            int rank = 0;
            for (int j = 0; j < p.B; ++j) {
                const int nj = qblocks(j);
                rank += (nj > ni) | ((nj == ni) & (j < i));
            }
            vtab->order[rank] = i;
        }
        __syncthreads();
        if (threadIdx.x == 0) {  // B <= 1024: a serial scan is a few microseconds at most
            int run = 0;
            for (int k = 0; k < p.B; ++k) {
                vtab->prefix[k] = run;
                const int nqb = qblocks(vtab->order[k]);
                run += p.Hq * (p.pair_tiles ? (nqb + 1) / 2 : nqb);
            }
            vtab->prefix[p.B] = run;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (vtab) {
        num_tiles = vtab->prefix[p.B];
        if (p.pair_tiles) {  // two members per pair, walked a grid-wide wave at a time
            const int g = (int)gridDim.x;
            num_tiles = 2 * g * ((num_tiles + g - 1) / g);
        }
    }
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

    if (warp == C::kProducerWarp) {
        // ------------------------------------------------------------ TMA producer --
        if (lane == 0) {
            uint32_t kv_it = 0, tcount = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileCoord c = decode_tile<C>(p, vtab, t);
                if (c.n_kv <= 0) continue;
                for (int q = 0; q < C::NQ && ok; ++q) {
                    ok = mbar_wait(bar(C::kBarQEmpty + q), (tcount & 1u) ^ 1u, wc);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(C::kBarQFull + q), C::kQBytes);
                    for (int a = 0; a < C::DA; ++a)
                        tma_load_4d(sQ + q * C::kQBytes + a * (C::BM * 128), &tm_q,
                                    bar(C::kBarQFull + q), a * 64, c.h, c.q_base + c.m0 + q * C::BM, c.tb);
                }
                for (int j = 0; j < c.n_kv && ok; ++j) {
                    const uint32_t st = kv_it % C::NS;
                    const uint32_t ph = ((kv_it / C::NS) & 1u) ^ 1u;
                    ok = mbar_wait(bar(C::kBarKEmpty + st), ph, wc);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar(C::kBarKFull + st), C::kKVBytes);
                    for (int a = 0; a < C::DA; ++a)
                        tma_load_4d(sK + st * C::kKVBytes + a * (C::BN * 128), &tm_k,
                                    bar(C::kBarKFull + st), a * 64, c.hk, c.k_base + (c.j0 + j) * C::BN, c.tb);
                    ok = mbar_wait(bar(C::kBarVEmpty + st), ph, wc);
                    if (!ok) {
                        // K of this iteration is in flight: account for it in the drain
                        mbar_wait_drain(bar(C::kBarKFull + st), (kv_it / C::NS) & 1u);
                        break;
                    }
                    mbar_arrive_expect_tx(bar(C::kBarVFull + st), C::kKVBytes);
                    for (int a = 0; a < C::DA; ++a)
                        tma_load_4d(sV + st * C::kKVBytes + a * (C::BN * 128), &tm_v,
                                    bar(C::kBarVFull + st), a * 64, c.hk, c.k_base + (c.j0 + j) * C::BN, c.tb);
                    ++kv_it;
                }
                ++tcount;
            }
            // Drain: every copy this warp started has landed before shared memory goes.
            // The last NS iterations hold the last use of each stage.
            for (uint32_t d = 0; d < (uint32_t)C::NS && d < kv_it; ++d) {
                const uint32_t last = kv_it - 1 - d;
                const uint32_t st = last % C::NS;
                mbar_wait_drain(bar(C::kBarKFull + st), (last / C::NS) & 1u);
                mbar_wait_drain(bar(C::kBarVFull + st), (last / C::NS) & 1u);
            }
            if (tcount > 0)
                for (int q = 0; q < C::NQ; ++q)
                    mbar_wait_drain(bar(C::kBarQFull + q), (tcount - 1) & 1u);
        }
        __syncwarp();
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------- MMA issuer ----
        // The whole warp runs this loop and one elected lane issues each tcgen05.mma and
        // tcgen05.commit: uniform control flow keeps the issue cheap, and the issue rate
        // is what feeds the tensor pipe.  Every lane waits on the barriers itself and the
        // outcome is voted, so the warp stays converged (elect.sync needs all 32 lanes)
        // even when a wait gives up.
        {
            constexpr uint32_t idesc_s = make_idesc_f16(128, C::BN, kBF16, false, false);
            constexpr uint32_t idesc_o = make_idesc_f16(128, C::D, kBF16, false, true);
            uint32_t kv_it = 0, tcount = 0, it = 0;
            bool ok = true;
            auto wait = [&](uint32_t b, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, parity, wc));
            };

            // Descriptors are built once; stepping K by 16 elements only advances the
            // start-address field in the low word, so each MMA issues with a constant
            // 32-bit add.
            const uint64_t dq = make_sdesc_sw128(sQ, 16, 1024);
            const uint64_t dk = make_sdesc_sw128(sK, 16, 1024);
            const uint64_t dv = make_sdesc_sw128(sV, C::BN * 128, 1024);
            const uint32_t q_lo = (uint32_t)dq, q_hi = (uint32_t)(dq >> 32);
            const uint32_t k_lo = (uint32_t)dk, k_hi = (uint32_t)(dk >> 32);
            const uint32_t v_lo = (uint32_t)dv, v_hi = (uint32_t)(dv >> 32);
            auto issue_s = [&](int q, uint32_t kst, uint32_t slot) {
                const uint32_t d = tmem + slot * C::BN;
                const uint32_t a = q_lo + (uint32_t)((q * C::kQBytes) >> 4);
                const uint32_t b = k_lo + ((kst * C::kKVBytes) >> 4);
                umma_ss_elect<false>(d, a, q_hi, b, k_hi, idesc_s);
#pragma unroll
                for (int kk = 1; kk < C::D / 16; ++kk)
                    umma_ss_elect<true>(d, a + (((kk >> 2) * (C::BM * 128) + (kk & 3) * 32) >> 4), q_hi,
                                        b + (((kk >> 2) * (C::BN * 128) + (kk & 3) * 32) >> 4), k_hi, idesc_s);
            };
            auto issue_pv = [&](int q, uint32_t vst, uint32_t slot, bool acc) {
                const uint32_t d = tmem + C::kOCol0 + q * C::D;
                const uint32_t a = C::kSAhead ? tmem + C::kPCol0 + q * (C::BN / 2) : tmem + slot * C::BN;
                const uint32_t b = v_lo + ((vst * C::kKVBytes) >> 4);
                if (acc)
                    umma_ts_elect<true>(d, a, b, v_hi, idesc_o);
                else
                    umma_ts_elect<false>(d, a, b, v_hi, idesc_o);
#pragma unroll
                for (int kk = 1; kk < C::BN / 16; ++kk)
                    umma_ts_elect<true>(d, a + kk * 8, b + ((kk * (16 * 128)) >> 4), v_hi, idesc_o);
            };
            auto slot_of = [&](int q, uint32_t iter) -> uint32_t {
                return C::NQ == 1 ? (iter & 1u) : (uint32_t)q;
            };

            // kSAhead issue order per tile: S_0(0) S_1(0), then for each block j
            // [S_0(j+1) S_1(j+1)] P.V_0(j) P.V_1(j).  S_q(j+1) waits until softmax q has
            // read S_q(j) (SFree); P.V_q(j) waits for P_q(j).  Every SFree phase is
            // awaited exactly once: the S issued after block `it` is that of block it + 1,
            // in this tile or as the first block of the next one.
            for (int t = blockIdx.x; C::kSAhead && t < num_tiles && ok; t += gridDim.x) {
                const TileCoord c = decode_tile<C>(p, vtab, t);
                const int n = c.n_kv;
                if (n <= 0) continue;
                for (int q = 0; q < C::NQ && ok; ++q) ok = wait(bar(C::kBarQFull + q), tcount & 1u);
                if (!ok) break;
                {
                    const uint32_t st = kv_it % C::NS;
                    ok = wait(bar(C::kBarKFull + st), (kv_it / C::NS) & 1u);
                    for (int q = 0; q < C::NQ && ok; ++q) {
                        if (it > 0) ok = wait(bar(C::kBarSFree + q), (it - 1) & 1u);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(q, st, (uint32_t)q);
                        umma_commit_elect(bar(C::kBarSFull + q));
                        if (n == 1) umma_commit_elect(bar(C::kBarQEmpty + q));
                    }
                    if (!ok) break;
                }
                for (int j = 0; j < n && ok; ++j) {
                    const uint32_t cur = kv_it + j;
                    const uint32_t st = cur % C::NS;
                    const uint32_t nst = (cur + 1) % C::NS;
                    if (j + 1 < n) {
                        ok = wait(bar(C::kBarKFull + nst), ((cur + 1) / C::NS) & 1u);
                        for (int q = 0; q < C::NQ && ok; ++q) {
                            ok = wait(bar(C::kBarSFree + q), it & 1u);
                            if (!ok) break;
                            tc_fence_after();
                            issue_s(q, nst, (uint32_t)q);
                            umma_commit_elect(bar(C::kBarSFull + q));
                            if (j + 2 == n) umma_commit_elect(bar(C::kBarQEmpty + q));
                        }
                        if (!ok) break;
                    }
                    ok = wait(bar(C::kBarVFull + st), (cur / C::NS) & 1u);
                    for (int q = 0; q < C::NQ && ok; ++q) {
                        ok = wait(bar(C::kBarPFull + q), it & 1u);
                        if (ok && j == 0 && tcount > 0)
                            ok = wait(bar(C::kBarODrained + q), (tcount - 1) & 1u);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(q, st, (uint32_t)q, j > 0);
                        umma_commit_elect(bar(C::kBarODone + q));
                    }
                    ++it;
                }
                kv_it += n;
                ++tcount;
            }
            for (int t = blockIdx.x; !C::kSAhead && t < num_tiles && ok; t += gridDim.x) {
                const TileCoord c = decode_tile<C>(p, vtab, t);
                const int n = c.n_kv;
                if (n <= 0) continue;
                for (int q = 0; q < C::NQ && ok; ++q) ok = wait(bar(C::kBarQFull + q), tcount & 1u);
                if (!ok) break;
                // Blocks fully masked for a sub-tile get no MMAs for it; its S-full barrier is
                // still committed (and its P-full still awaited) so every phase stays in step.
                int blo[C::NQ], bhi[C::NQ];
#pragma unroll
                for (int q = 0; q < C::NQ; ++q) {
                    blo[q] = 0;
                    bhi[q] = n - 1;
                    if (kSkip) sub_tile_blocks<C>(p, c, q, blo[q], bhi[q]);
                }
                auto live = [&](int q, int j) -> bool { return !kSkip || (j >= blo[q] && j <= bhi[q]); };
                {
                    const uint32_t st = kv_it % C::NS;
                    // TMA-filled operands need no tcgen05 fence: the mbarrier wait orders them.
                    ok = wait(bar(C::kBarKFull + st), (kv_it / C::NS) & 1u);
                    if (!ok) break;
                    for (int q = 0; q < C::NQ; ++q) {
                        if (live(q, 0)) issue_s(q, st, slot_of(q, it));
                        umma_commit_elect(bar(C::kBarSFull + slot_of(q, it)));
                    }
                    if (!C::kRingBySoftmax) umma_commit_elect(bar(C::kBarKEmpty + st));
                    if (n == 1)
                        for (int q = 0; q < C::NQ; ++q) umma_commit_elect(bar(C::kBarQEmpty + q));
                }
                for (int j = 0; j < n && ok; ++j) {
                    const uint32_t cur = kv_it + j;
                    const uint32_t st = cur % C::NS;
                    const uint32_t nst = (cur + 1) % C::NS;
                    const bool more = (j + 1 < n);
                    if (C::NQ == 1 && more) {
                        ok = wait(bar(C::kBarKFull + nst), ((cur + 1) / C::NS) & 1u);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(0, nst, slot_of(0, it + 1));
                        umma_commit_elect(bar(C::kBarSFull + slot_of(0, it + 1)));
                        umma_commit_elect(bar(C::kBarKEmpty + nst));
                        if (j + 2 == n) umma_commit_elect(bar(C::kBarQEmpty + 0));
                    }
                    ok = wait(bar(C::kBarVFull + st), (cur / C::NS) & 1u);
                    if (!ok) break;
                    for (int q = 0; q < C::NQ && ok; ++q) {
                        ok = wait(bar(C::kBarPFull + q), it & 1u);
                        if (ok && j == 0 && tcount > 0)
                            ok = wait(bar(C::kBarODrained + q), (tcount - 1) & 1u);
                        if (!ok) break;
                        tc_fence_after();
                        // the sub-tile's first live block initialises O
                        if (live(q, j)) issue_pv(q, st, slot_of(q, it), j > (kSkip ? blo[q] : 0));
                        if (kOPerIter || j + 1 == n) umma_commit_elect(bar(C::kBarODone + q));
                        if (C::NQ > 1 && more) {
                            if (q == 0) {
                                ok = wait(bar(C::kBarKFull + nst), ((cur + 1) / C::NS) & 1u);
                                if (!ok) break;
                            }
                            if (live(q, j + 1)) issue_s(q, nst, slot_of(q, it + 1));
                            umma_commit_elect(bar(C::kBarSFull + slot_of(q, it + 1)));
                            if (!C::kRingBySoftmax && q == C::NQ - 1)
                                umma_commit_elect(bar(C::kBarKEmpty + nst));
                            if (j + 2 == n) umma_commit_elect(bar(C::kBarQEmpty + q));
                        }
                    }
                    if (!ok) break;
                    if (!C::kRingBySoftmax) umma_commit_elect(bar(C::kBarVEmpty + st));
                    ++it;
                }
                kv_it += n;
                ++tcount;
            }
            // Every MMA issued has completed before TMEM and shared memory are released.
            umma_commit_elect(bar(C::kBarFinal));
            mbar_wait_drain(bar(C::kBarFinal), 0);
            __syncwarp();
        }
    } else if (warp == C::kStoreWarp) {
        // ---------------------------------------------------------- O store warp ----
        // The staging buffer's uses are the rounds of the Q sub-tiles, in the order (tile
        // with keys, sub-tile q, round).  The buffer is handed from use to use: the
        // warpgroup of use u fills it and arrives on Staged; this warp waits for Staged,
        // stores, and once the store has read the buffer passes it on by arriving on the
        // StageFree barrier of use u + 1's warpgroup.  Use 0 belongs to warpgroup 0, which
        // starts out holding the buffer.  Each StageFree barrier has one waiter and completes one phase per
        // use of its warpgroup after that warpgroup's previous one was read, so its parity
        // waits are exact; Staged cannot run ahead of this warp either.
        if (!kVarlen && lane == 0) {
            uint32_t use = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileCoord c = decode_tile<C>(p, vtab, t);
                if (c.n_kv <= 0) continue;
                for (int q = 0; q < C::NQ && ok; ++q) {
                    for (int rd = 0; rd < L::kStageRounds; ++rd) {
                        if (use > 0) mbar_arrive(bar(C::kBarStageFree + q));  // the buffer is q's
                        ok = mbar_wait(bar(C::kBarStaged), use & 1u, wc);
                        if (!ok) break;
                        // a box whose first row is past the sequence holds nothing to store
                        if (c.m0 + q * C::BM < c.sq)
                            for (int a = 0; a < L::kStageAtoms; ++a)
                                tma_store_4d(&tm_o, sStage + a * (C::BM * 128), (rd * L::kStageAtoms + a) * 64,
                                             c.h, c.q_base + c.m0 + q * C::BM, c.tb);
                        bulk_commit_group();
                        bulk_wait_read_all();
                        ++use;
                    }
                }
            }
            bulk_wait_all();  // every store has landed before the kernel ends
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ softmax warpgroups ----
        const int q = warp >> 2;
        const int wq = warp & 3;           // TMEM lane quadrant of this warp
        const int r = wq * 32 + lane;      // row within the 128-row Q tile
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const uint32_t tO = lane_base + C::kOCol0 + q * C::D;
        const float kNegInf = -__int_as_float(0x7f800000);
        constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8
        constexpr int kSC = C::BN / 32;        // 32-column chunks of S per block
        const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
        uint32_t it = 0, tcount = 0;
        uint32_t nstaged = 0;  // staging-buffer uses of this warpgroup so far
        bool ok = true;

        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const TileCoord c = decode_tile<C>(p, vtab, t);
            const int row = c.m0 + q * C::BM + r;
            const int off = c.sk - c.sq;  // bottom-right causal alignment
            // Rows are stored only inside the sequence and inside the packed tensor (the
            // second test guards against malformed cu_seqlens of a variable-length batch).
            const bool row_ok = row < c.sq && c.o_row0 + row >= 0 && c.o_row0 + row < p.total_q;
            const size_t o_row = (size_t)(c.o_row0 + row) * p.Hq + c.h;
            uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + o_row * C::D;
            if (c.n_kv < 0) continue;  // not a tile (causal pairing)
            if (c.n_kv == 0) {
                if (row_ok) {
#pragma unroll
                    for (int d = 0; d < C::D; d += 8) st_global_v4(orow + d, 0u, 0u, 0u, 0u);
                    if (p.lse) p.lse[c.lse0 + row] = kNegInf;
                }
                continue;
            }
            float m_run = kNegInf;  // running max, log2 units (raw score * scale * log2 e)
            uint64_t l2 = f2_pack(0.f, 0.f);  // running sum, two interleaved partial sums
            const int tile_row0 = c.m0 + q * C::BM;
            int blo = 0, bhi = c.n_kv - 1;  // this sub-tile's live blocks (kSkip: others skipped)
            if (kSkip) sub_tile_blocks<C>(p, c, q, blo, bhi);

            for (int j = 0; j < c.n_kv; ++j) {
                const uint32_t slot = (C::NQ == 1) ? (it & 1u) : (uint32_t)q;
                const uint32_t spar = (C::NQ == 1) ? ((it >> 1) & 1u) : (it & 1u);
                ok = mbar_wait(bar(C::kBarSFull + slot), spar, wc);
                if (!ok) break;
                tc_fence_after();
                if (C::kRingBySoftmax && q == C::NQ - 1 && wq == 0 && lane == 0) {
                    mbar_arrive(bar(C::kBarKEmpty + it % C::NS));  // K of this block
                    if (it >= C::kVReleaseLag)  // V of an earlier block
                        mbar_arrive(bar(C::kBarVEmpty + (it - C::kVReleaseLag) % C::NS));
                }
                if (kSkip && (j < blo || j > bhi)) {  // fully masked for this sub-tile: no S
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::kBarPFull + q));
                    ++it;
                    continue;
                }
                const uint32_t tS = lane_base + slot * C::BN;
                // P goes over S, or into its own columns with kSAhead.
                const uint32_t tP = C::kSAhead ? lane_base + C::kPCol0 + q * (C::BN / 2) : tS;
                // All chunks of S are loaded before a single wait.
                uint32_t u[kSC][32];
#pragma unroll
                for (int ch = 0; ch < kSC; ++ch) tmem_ld_32x32b_x32(tS + ch * 32, u[ch]);
                tmem_wait_ld(u[0]);
#pragma unroll
                for (int ch = 1; ch < kSC; ++ch) reg_fence(u[ch]);
                if (C::kSAhead) {  // S is in registers: the next S of this tile may be issued
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::kBarSFree + q));
                }

                const int n0 = (c.j0 + j) * C::BN;
                const bool need_mask =
                    (n0 + C::BN > c.sk) ||
                    (p.has_hi && (n0 + C::BN - 1 > tile_row0 + off + p.hi_off)) ||
                    (p.has_lo && (n0 < tile_row0 + C::BM - 1 + off - p.win_left));
                // Two ways to mask (both exact).  The general fixed-length kernels compare
                // and select per score on the integer pipe.  The others (sliding windows,
                // packed variable-length batches, S ahead of P.V) add 2^126 times a mask
                // bit t (1: masked) that one saturating add computes on the FMA pipe: s -
                // 2^126 is about -2^126 for any finite s, and its exponential 0.  The column
                // and the bounds (clamped to [-1, BN]) are small integers, so t is exactly 0
                // or 1.  A row with every score of the block masked then has no maximum here.
                constexpr bool kFmaMask = kSkip || kVarlen || C::kSAhead;
                if (need_mask) {
                    int kmax = c.sk - 1 - n0;
                    if (p.has_hi) kmax = min(kmax, row + off + p.hi_off - n0);
                    constexpr float kS = 18446744073709551616.0f;    // 2^64
                    constexpr float kOut = -8.5070591730234616e37f;  // -2^126
                    // (the window instantiation always has a lower bound, and keeps the one loop)
                    if (kSkip || p.has_lo) {
                        const int kmin = p.has_lo ? row + off - p.win_left - n0 : -1;
                        if constexpr (kFmaMask) {
                            // masked iff |col - mid| > half the width of [kmin, kmax]
                            const float lo = (float)min(max(kmin, -1), C::BN), hi = (float)min(max(kmax, -1), C::BN);
                            const float mid = (lo + hi) * (0.5f * kS);
                            const float half = ((hi - lo) * 0.5f + 0.5f) * kS;
#pragma unroll
                            for (int ch = 0; ch < kSC; ++ch)
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    const float t = __saturatef(fabsf((float)(ch * 32 + i) * kS - mid) - half);
                                    u[ch][i] = __float_as_uint(fmaf(t, kOut, __uint_as_float(u[ch][i])));
                                }
                        } else {
#pragma unroll
                            for (int ch = 0; ch < kSC; ++ch)
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    u[ch][i] = ((ch * 32 + i > kmax) | (ch * 32 + i < kmin)) ? 0xff800000u : u[ch][i];
                        }
                    } else {  // no lower bound: masked iff col > kmax
                        if constexpr (kFmaMask) {
                            const float edge = ((float)min(max(kmax, -1), C::BN) + 0.5f) * kS;
#pragma unroll
                            for (int ch = 0; ch < kSC; ++ch)
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    const float t = __saturatef((float)(ch * 32 + i) * kS - edge);
                                    u[ch][i] = __float_as_uint(fmaf(t, kOut, __uint_as_float(u[ch][i])));
                                }
                        } else {
#pragma unroll
                            for (int ch = 0; ch < kSC; ++ch)
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    u[ch][i] = (ch * 32 + i > kmax) ? 0xff800000u : u[ch][i];
                        }
                    }
                }
                // Row max over the BN scores: four independent chains of 3-input maxima.
                auto sv = [&](int k) -> float { return __uint_as_float(u[k >> 5][k & 31]); };
                float mx[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) mx[k] = sv(k);
#pragma unroll
                for (int k = 4; k + 8 <= C::BN; k += 8)
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) mx[c4] = max3f(mx[c4], sv(k + c4), sv(k + c4 + 4));
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) mx[c4] = fmaxf(mx[c4], sv(C::BN - 4 + c4));
                const float raw_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                const float m_blk =
                    (kFmaMask && raw_max < -4.2535295865117308e37f) ? kNegInf : raw_max * p.scale_log2;
                const bool bump = m_blk > m_run + kRescaleLog2;
                const float m_new = bump ? m_blk : m_run;
                const float alpha = bump ? ex2_approx(m_run - m_new) : 1.0f;
                m_run = m_new;
                const float m_sub = (m_run == kNegInf) ? 0.f : m_run;
                const uint64_t nm2 = f2_pack(-m_sub, -m_sub);

                // P = exp2(s * scale * log2 e - m), rounded to 16 bits and written to TMEM
                // (over S, or into P's own columns), 32 columns at a time.  With kSAhead the
                // P columns and O are still read by P.V of the previous block: all of P is
                // computed first, then that P.V is awaited, then P is stored.
                uint64_t sum2 = f2_pack(0.f, 0.f);
                uint32_t pk[kSC][16];
#pragma unroll
                for (int ch = 0; ch < kSC; ++ch) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint64_t a = fma2(f2_pack(__uint_as_float(u[ch][2 * i]),
                                                        __uint_as_float(u[ch][2 * i + 1])),
                                                c2, nm2);
                        float a0, a1;
                        f2_unpack(a, a0, a1);
                        const float p0 = ex2_approx(a0);
                        const float p1 = ex2_approx(a1);
                        sum2 = add2(sum2, f2_pack(p0, p1));
                        pk[ch][i] = pack2<kBF16>(p0, p1);
                    }
                    if (!C::kSAhead) tmem_st_32x32b_x16(tP + ch * 16, pk[ch]);
                }
                l2 = fma2(l2, f2_pack(alpha, alpha), sum2);
                if (C::kSAhead) {
                    if (j > 0) {
                        ok = mbar_wait(bar(C::kBarODone + q), (it - 1) & 1u, wc);
                        if (!ok) break;
                        tc_fence_after();
                    }
#pragma unroll
                    for (int ch = 0; ch < kSC; ++ch) tmem_st_32x32b_x16(tP + ch * 16, pk[ch]);
                }

                if (C::NQ == 1 && j > 0) {
                    // NQ == 1: the next S is issued ahead of the previous P.V, so that P.V's
                    // completion is awaited here before O may be rescaled.
                    ok = mbar_wait(bar(C::kBarODone + q), (it - 1) & 1u, wc);
                    if (!ok) break;
                    tc_fence_after();
                }
                // NQ == 2: S of this block was issued after the previous P.V of this tile,
                // so its completion (awaited above) implies that P.V has completed; with
                // kSAhead that P.V was awaited before the P stores.
                if (j > (kSkip ? blo : 0) && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
                    for (int ch = 0; ch < C::D / 32; ++ch) {
                        uint32_t ov[32];
                        tmem_ld_32x32b_x32(tO + ch * 32, ov);
                        tmem_wait_ld(ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st_32x32b_x32(tO + ch * 32, ov);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarPFull + q));
                ++it;
            }
            if (!ok) break;

            // ------------------------------------------------------------ epilogue ----
            ok = mbar_wait(bar(C::kBarODone + q), kOPerIter ? ((it - 1) & 1u) : (tcount & 1u), wc);
            if (!ok) break;
            tc_fence_after();
            ++tcount;
            float l0, l1;
            f2_unpack(l2, l0, l1);
            const float l_run = l0 + l1;
            const float inv_l = (l_run > 0.f) ? 1.0f / l_run : 0.f;
            // O goes through the staging buffer in the TMA layout (128-byte swizzle: 16-byte
            // chunk k of row r sits at chunk k ^ (r % 8)) and the store warp writes it; rows
            // past Sq are clipped by the tensor map.  Sub-tiles that are not staged (partial
            // ones of a packed variable-length batch) store their rows directly.
            constexpr bool use_stage = !kVarlen;
            // The i-th use of this warpgroup waits for phase i of its StageFree barrier
            // (phase i - 1 for warpgroup 0, which holds the buffer before use 0).
            auto stage_wait = [&]() -> bool {
                const int ph = (int)nstaged - (q == 0 ? 1 : 0);
                ++nstaged;
                return ph < 0 || mbar_wait(bar(C::kBarStageFree + q), (uint32_t)ph & 1u, wc);
            };
            auto stage_done = [&]() {
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarStaged));
            };
            // 32 columns of this row (from TMEM, fp32) -> bf16/fp16, into the staging buffer
            // or out to global memory.  col is the first column within the row.
            auto put_chunk = [&](int col, const uint32_t (&ov)[32]) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)  // kSkip: a sub-tile that saw no key left O unwritten
                    w[i] = pack2<kBF16>(kSkip && !(inv_l > 0.f) ? 0.f : __uint_as_float(ov[2 * i]) * inv_l,
                                        kSkip && !(inv_l > 0.f) ? 0.f : __uint_as_float(ov[2 * i + 1]) * inv_l);
                if (use_stage) {
                    const int sc = col % (L::kStageAtoms * 64);  // column within the staged round
                    const uint32_t rowb = sStage + (uint32_t)(sc / 64) * (C::BM * 128) + (uint32_t)r * 128;
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        const uint32_t k16 = (uint32_t)((sc % 64) / 8 + v4);
                        st_shared_v4(rowb + ((k16 ^ (uint32_t)(r & 7)) << 4), w[4 * v4], w[4 * v4 + 1],
                                     w[4 * v4 + 2], w[4 * v4 + 3]);
                    }
                } else if (row_ok) {
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        st_global_v4(orow + col + v4 * 8, w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2],
                                     w[4 * v4 + 3]);
                }
            };
            constexpr int kChunksPerRound = L::kStageAtoms * 2;  // 32-column chunks per round
            if constexpr (C::D <= 128) {
                // All of O comes out of TMEM behind one wait and the accumulator is handed
                // back before the normalisation and the stores, so the next tile's first P.V
                // does not wait for them.
                uint32_t ov[C::D / 32][32];
#pragma unroll
                for (int ch = 0; ch < C::D / 32; ++ch) tmem_ld_32x32b_x32(tO + ch * 32, ov[ch]);
                tmem_wait_ld(ov[0]);
#pragma unroll
                for (int ch = 1; ch < C::D / 32; ++ch) reg_fence(ov[ch]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarODrained + q));
#pragma unroll
                for (int ch = 0; ch < C::D / 32; ++ch) {
                    if (use_stage && ch % kChunksPerRound == 0) {
                        ok = stage_wait();
                        if (!ok) break;
                    }
                    put_chunk(ch * 32, ov[ch]);
                    if (use_stage && (ch % kChunksPerRound == kChunksPerRound - 1 || ch == C::D / 32 - 1))
                        stage_done();
                }
                if (!ok) break;
            } else {
                // Wide tiles: 32 columns at a time, staged in rounds.
#pragma unroll
                for (int ch = 0; ch < C::D / 32; ++ch) {
                    if (use_stage && ch % kChunksPerRound == 0) {
                        ok = stage_wait();
                        if (!ok) break;
                    }
                    uint32_t ov[32];
                    tmem_ld_32x32b_x32(tO + ch * 32, ov);
                    tmem_wait_ld(ov);
                    put_chunk(ch * 32, ov);
                    if (use_stage && (ch % kChunksPerRound == kChunksPerRound - 1 || ch == C::D / 32 - 1))
                        stage_done();
                }
                if (!ok) break;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarODrained + q));
            }
            if (p.lse && row_ok) {
                const float lse = (l_run > 0.f) ? (m_run + lg2_approx(l_run)) * 0.69314718055994531f
                                                : kNegInf;
                p.lse[c.lse0 + row] = lse;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Causal tile walk: whether pairing long and short query blocks (FwdParams::pair_tiles)
// leaves the busiest CTA less work than dealing the blocks out longest first.  Query block
// qb of a head covers about qb + 1 of its key spans; each tile also costs about half a
// span of fixed overhead.  Both walks are replayed, over up to 2^18 tiles; beyond that
// many tiles per CTA even out either way and pairing is kept.
inline bool causal_pairs_balance_better(long long heads, int nqb, int sms) {
    const long long tiles = heads * nqb;
    const long long pairs = heads * ((nqb + 1) / 2);
    if (tiles > (1LL << 18) || sms > 1024) return true;
    const int g_rr = (int)(tiles < sms ? tiles : sms);
    const int g_pr = (int)(pairs < sms ? pairs : sms);
    static thread_local long long load[1024];
    for (int i = 0; i < g_rr; ++i) load[i] = 0;
    for (long long t = 0; t < tiles; ++t) load[t % g_rr] += 2 * (nqb - (t % nqb)) + 1;
    long long max_rr = 0;
    for (int i = 0; i < g_rr; ++i) max_rr = load[i] > max_rr ? load[i] : max_rr;
    for (int i = 0; i < g_pr; ++i) load[i] = 0;
    const int per = (nqb + 1) / 2;
    for (long long v = 0; v < pairs; ++v) {
        const int k = (int)(v % per);
        long long w = 2 * (nqb - k) + 1;             // the long block, qb = nqb - 1 - k
        if (nqb - 1 - k != k) w += 2 * (k + 1) + 1;  // the short one, qb = k
        load[v % g_pr] += w;
    }
    long long max_pr = 0;
    for (int i = 0; i < g_pr; ++i) max_pr = load[i] > max_pr ? load[i] : max_pr;
    return max_pr < max_rr;
}

// Host launcher for one configuration.
template <class C>
fa_status launch_fwd_cfg(const FwdArgs& a, cudaStream_t stream) {
    static int attr_bf16[64] = {0};
    static int attr_f16[64] = {0};
    static int attr_bf16_v[64] = {0};
    static int attr_f16_v[64] = {0};
    static int attr_bf16_s[64] = {0};
    static int attr_f16_s[64] = {0};
    CUtensorMap tq, tk, tv, to;
    const bool varlen = a.cu_q != nullptr;
    // Fixed-length batches map [B, S, H, D] as (D, H, S, B); packed variable-length
    // batches map [total, H, D] as (D, H, total, 1).
    const uint64_t q_rows = varlen ? (uint64_t)a.total_q : (uint64_t)a.Sq;
    const uint64_t k_rows = varlen ? (uint64_t)a.total_k : (uint64_t)a.Sk;
    const uint64_t outer = varlen ? 1 : (uint64_t)a.B;
    if (!encode_tmap_4d(&tq, a.q, a.bf16, a.D, a.Hq, q_rows, outer, C::BM) ||
        !encode_tmap_4d(&tk, a.k, a.bf16, a.D, a.Hkv, k_rows, outer, C::BN) ||
        !encode_tmap_4d(&tv, a.v, a.bf16, a.D, a.Hkv, k_rows, outer, C::BN))
        return FA_ERR_CUDA;
    // O is written by TMA stores of 128-row boxes (of packed rows for a variable-length batch).
    if (!encode_tmap_4d(&to, a.o, a.bf16, a.D, a.Hq, q_rows, outer, C::BM)) return FA_ERR_CUDA;
    FwdParams p;
    p.B = a.B;
    p.Sq = a.Sq;
    p.Sk = a.Sk;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.group = a.Hq / a.Hkv;
    p.causal = a.causal ? 1 : 0;
    p.has_lo = a.window_left >= 0 ? 1 : 0;
    p.win_left = a.window_left >= 0 ? a.window_left : 0;
    p.has_hi = (a.causal || a.window_right >= 0) ? 1 : 0;
    p.hi_off = a.causal ? 0 : (a.window_right >= 0 ? a.window_right : 0);
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.pair_tiles = 0;
    p.cu_q = a.cu_q;
    p.cu_k = a.cu_k;
    p.total_q = varlen ? a.total_q : a.B * a.Sq;  // packed rows of O (the store guard)
    int grid = a.num_sms;
    if (!varlen) {
        p.num_qb = (a.Sq + C::NQ * C::BM - 1) / (C::NQ * C::BM);
        const long long tiles = (long long)a.B * a.Hq * p.num_qb;
        if (tiles > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
        p.num_tiles = (int)tiles;
        grid = p.num_tiles < a.num_sms ? p.num_tiles : a.num_sms;
        if (a.causal && a.window_left < 0 && p.num_qb > 1 &&
            causal_pairs_balance_better((long long)a.B * a.Hq, p.num_qb, a.num_sms)) {
            // causal: query blocks go out in long/short pairs, one pair per CTA at a time
            const long long pairs = (long long)a.B * a.Hq * ((p.num_qb + 1) / 2);
            grid = pairs < a.num_sms ? (int)pairs : a.num_sms;
            const long long walked = 2LL * grid * ((pairs + grid - 1) / grid);
            if (walked > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
            p.num_tiles = (int)walked;
            p.pair_tiles = 1;
        }
    } else {
        p.num_qb = 0;
        p.num_tiles = 0;  // counted on the device from cu_seqlens
        // causal: pair long and short query blocks of each (sequence, head)
        p.pair_tiles = (a.causal && a.window_left < 0) ? 1 : 0;
    }
    p.o = a.o;
    p.lse = a.lse;
    p.status = a.dev_status;
    auto kern = varlen ? (a.bf16 ? fa_fwd_kernel<C, true, true> : fa_fwd_kernel<C, false, true>)
                       : (a.bf16 ? fa_fwd_kernel<C, true, false> : fa_fwd_kernel<C, false, false>);
    // Fixed-length sliding windows take the instantiation that skips a sub-tile's blocks
    // outside its window (two Q tiles with P over S only).
    bool skip = false;
    if constexpr (C::NQ == 2 && !C::kSAhead) {
        if (!varlen && a.window_left >= 0) {
            kern = a.bf16 ? fa_fwd_kernel<C, true, false, true> : fa_fwd_kernel<C, false, false, true>;
            skip = true;
        }
    }
    const int smem = varlen ? C::template Layout<true>::kSmemBytes : C::template Layout<false>::kSmemBytes;
    int* flags = varlen ? (a.bf16 ? attr_bf16_v : attr_f16_v)
                        : skip ? (a.bf16 ? attr_bf16_s : attr_f16_s) : (a.bf16 ? attr_bf16 : attr_f16);
    if (!ensure_smem_attr((const void*)kern, smem, flags)) return FA_ERR_CUDA;
    kern<<<grid, C::kThreads, smem, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
