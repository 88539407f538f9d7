// sift_attention.cu -- block-sparse (and dense) causal grouped-query flash
// attention for SIFT's online prefill on sm_103a.
//
// SIFT pages (gist.science/it/paper/2606.09441), "Dettagli di
// Implementazione": the sparse attention kernel iterates only over the tile
// indices decoded from the bit vectors; "Esecuzione Online": flagged tiles are
// computed, the rest skipped.  The pages' kernel extends FlashAttention-3 on
// H200; this one is written for Blackwell: TMA tile loads, tcgen05 MMAs with
// the accumulators in tensor memory, and a persistent longest-first scheduler.
//
// One work item = (query tile i, kv head h, pair of query heads of h's group).
// Both heads of the pair share every K/V tile staged in shared memory, and the
// decoded list of row (h, i).  Roles inside the CTA (384 threads; 352 on the general
// layout, which has no warp 11):
//   warps 0-3  softmax of head slot 0 (thread = query row = TMEM lane); after the item's
//              last tile, its epilogue: O / l in bf16 into the shared-memory staging tile
//              (general layout: straight to global memory, row by row)
//   warps 4-7  softmax of head slot 1, the same, staging into the V ring slot of the
//              item's last V tile instead (free once P*V is done)
//   warp  8    scheduler + K producer (K_j into a ring of 2 slots, 3 on the general
//              layout); it claims the next item early and runs ahead into its K tiles
//   warp  9    TMEM allocator + MMA issuer (warp-wide loop, one elected lane issues)
//   warp 10    Q + V producer (the item's Q pair once the previous one is released, then
//              V_j into a 2-slot ring; for rows walked from the bits it takes warp 8's
//              tile coordinates from a shared-memory ring instead of walking them again)
//   warp 11    O writer: one TMA store per staged head tile, then hands the staging tile
//              back to head 0, and the V slot to the V producer, once the store has read it
// Tensor memory (128 lanes x 512 columns): S_0 | S_1 | O_0 | O_1, 128 columns
// each.  P (bf16, two per column) overwrites the first half of its S, and the
// P*V MMA reads it from tensor memory, so P never touches shared memory.
// MMA order per item: S0(0) S1(0) | PV0(0) S0(1) | PV1(0) S1(1) | ... so the
// tensor pipe works on one head while the other head's softmax runs.  Each P
// reaches the issuer in two halves of the keys, each on a barrier of its own,
// so P*V over the first half runs while the softmax finishes the second.
// Online softmax keeps a per-row running max m (log2 units) and sum l; O is
// rescaled only when m grows by more than 8 (factor 256) -- otherwise the
// stale max is kept, which stays exact because O and l share it.  The rescale
// comes before the tile's first half of P is handed over.
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records
// SIFT_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <climits>
#include <type_traits>
#include <mutex>

#include "ptx.cuh"
#include "sift_internal.h"

namespace sift {
namespace {

// threads of a CTA: 12 warps, or 11 on the general layout (no O writer)
constexpr int threads_for(bool staged) { return staged ? 384 : 352; }
constexpr int kProducerWarp = 8;   // scheduler and K loads
constexpr int kMmaWarp = 9;        // TMEM allocator and MMA issuer
constexpr int kVProducerWarp = 10; // Q and V loads
constexpr int kStoreWarp = 11;     // TMA stores of O
// K ring: three slots on the general layout; two elsewhere, where the shared memory of the
// third holds the staging tile of O instead (measured on aligned rows: the third K slot
// was worth nothing, the staged O stores 1.5%; on the general layout, whose gathered pages
// keep the copy engine busier, the TMA stores cost 5%).  V ring: two slots.
constexpr int kKSlotsMax = 3;
constexpr int kVSlots = 2;
constexpr int kRing = 16;  // key tiles in flight from the K producer to the V producer (bits)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kMinSmem = 120 * 1024;  // forces one CTA per SM (the CTA owns all of TMEM)

// where a work item's key-tile list comes from
constexpr int kModeList = 0;   // decoded lists in HBM (sift_sparse_prefill)
constexpr int kModeDense = 1;  // implicit {prompt start .. i} (sift_dense_prefill)
constexpr int kModeBits = 2;   // the LA/CA bits themselves, walked on the fly (sift_fused_prefill)
constexpr int kModeRagged = 3; // (first token, info) lists of a general layout (sift_sparse_prefill_ragged)
constexpr int kMaxFusedPrompts = 64;

struct WorkItem {
    int32_t valid;
    int32_t h;      // kv head
    int32_t i;      // global query tile
    int32_t hq0;    // first query head of the pair
    int32_t n;      // key tiles in the row's list
    int32_t first;  // dense rows: first tile of the prompt
    int64_t list;   // sparse rows: element offset of the row inside the kv_idx slice
    // rows walked from the bits
    int32_t pt;      // first tile of the prompt
    int32_t g;       // the row's document, -1 for a suffix row
    int32_t g0;      // first document of the prompt
    int32_t t0;      // first tile of the row's document
    int32_t W;       // LA words per row of the document
    int32_t pad;
    int64_t la_row;  // word offset of the row's LA words
    // general layout: the query tile's first token and its rows inside the segment
    int32_t q0, qlen;
};

struct Ctl {
    // per head slot: a slot's Q for the next item loads as soon as this item's last S of
    // that head is done (head 0's a step before head 1's)
    uint64_t q_full[2], q_empty[2];
    uint64_t k_full[kKSlotsMax], k_empty[kKSlotsMax], v_full[kVSlots], v_empty[kVSlots];
    // p_half[s]: the first half of head s's P (keys [0, B/2)) is in tensor memory
    uint64_t s_full[2], p_half[2], p_full[2], o_full[2];
    // O staging: head 0 writes the staging tile, head 1 the V ring slot of the item's last
    // V tile; stage_full[s] when head s has written its tile, stage_free[0] when the TMA
    // store of head 0's tile has read it (head 1's slot goes back through v_empty)
    uint64_t stage_full[2], stage_free[2];
    uint64_t sch_full[2], sch_empty[2];
    uint64_t teardown, never;
    // rows walked from the bits: the K producer hands each key tile it finds to the V
    // producer (entry t % kRing of tile t, complete once written); the V producer trails
    // by a few tiles at most, since S(j) is issued only after V(j-1) has landed
    uint64_t ring_full[kRing];
    int32_t ring[kRing];
    WorkItem items[2];
    uint32_t tmem_base;
    volatile int32_t abort;
    // rows walked from the bits: prompts by decreasing length (rank -> prompt, tiles)
    int32_t pord[kMaxFusedPrompts];
    int32_t plen[kMaxFusedPrompts];
};

struct AttnParams {
    const int32_t *kv_idx;  // layer slice [Hkv][N][rowcap] (sparse)
    const int32_t *counts;  // [U]
    const int32_t *sched;   // [U]
    __nv_bfloat16 *o;
    float *lse;
    int32_t *work_counter;
    int32_t *status;
    int32_t total_items, U, N, Hq, G, pairs, rowcap, total_tokens;
    float scale_log2;
    uint64_t timeout_ns;
    int32_t stall;
    // rows walked from the bits (sift_fused_prefill)
    const int32_t *cu, *doc_cu, *doc_end;
    const int64_t *la_off, *ca_off;
    const uint64_t *la, *ca;
    int64_t la_len, ca_len;
    int32_t P, D, B, layer, Hkv;
    // general layout (sift_sparse_prefill_ragged)
    const int2 *kv2;         // layer slice [Hkv][NQ][rowcap] of (first token, info)
    const int32_t *qt;       // [NQ][2] (first token, rows)
    int32_t lp;              // log2 of min(page, tile)
    uint32_t full_info;      // info of a whole tile with every page kept
    const int32_t *pages;    // gathered pages: layer slice [Hkv][D][page_cap] of first tokens
    int64_t pages_len;       // entries in that slice
    int32_t page;            // page size in tokens (gathered loads are page rows high)
    int32_t o_v8;            // o is 32-byte aligned: the epilogue writes whole sectors
};

constexpr uint32_t kGatherBit = 1u << 9;  // list entry of gathered pages (general layout)

template <int BT, int HD, bool STAGED>
struct Geo {
    static constexpr int kKSlots = STAGED ? 2 : 3;
    static constexpr int kBoxes = HD / 64;          // 64-column (128-byte) swizzled boxes
    static constexpr int kQBox = 128 * 128;          // bytes: 128 rows (MMA M) x 128 B
    static constexpr int kQBytes = 2 * kBoxes * kQBox;
    static constexpr int kKVBox = BT * 128;
    static constexpr int kKVBytes = kBoxes * kKVBox;
    static constexpr int kKOff = kQBytes;
    static constexpr int kVOff = kKOff + kKSlots * kKVBytes;
    static constexpr int kOBox = BT * 128;                 // bytes: tile rows x 128 B
    static constexpr int kOOff = kVOff + kVSlots * kKVBytes;  // O staging tile, kBoxes boxes
    static constexpr int kCtlOff = kOOff + (STAGED ? kBoxes * kOBox : 0);
    static constexpr int kSmemUsed = kCtlOff + 1536 + 1024;  // + control block + align slack
    static constexpr int kSmem = kSmemUsed > kMinSmem ? kSmemUsed : kMinSmem;
    static constexpr uint32_t kTxQ = 2 * kBoxes * BT * 128;
    static constexpr uint32_t kTxKV = kBoxes * BT * 128;
    static constexpr int kSoftWarps = BT / 32;       // active softmax warps per head slot
    static constexpr uint32_t kIdescS = ptx::idesc_bf16(128, BT, false, false);
    static constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, HD, false, true);
    static_assert(sizeof(Ctl) <= 1536, "control block");
    static_assert(kSmemUsed <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void set_status(int32_t *st, int code) { atomicCAS(st, 0, code); }

// bounded wait; gives up early once another role has aborted
__device__ __noinline__ bool wait_bar(Ctl &c, uint32_t bar, uint32_t parity, uint64_t timeout,
                                      int32_t *status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (c.abort) return false;
        if (ptx::globaltimer_ns() - t0 > timeout) {
            c.abort = 1;
            set_status(status, SIFT_ERR_TIMEOUT);
            return false;
        }
    }
}

// bounded wait used while unwinding (ignores the abort flag)
__device__ __noinline__ bool drain_bar(uint32_t bar, uint32_t parity, uint64_t timeout) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer_ns() - t0 > timeout) return false;
    return true;
}

// bounded wait with an inlined fast path for a phase that has already completed (a
// call into the slow path costs hundreds of cycles on the MMA issuer's critical path)
__device__ __forceinline__ bool wait1(Ctl &c, uint32_t bar, uint32_t parity, const AttnParams &p) {
    return ptx::mbar_test_wait(bar, parity) || wait_bar(c, bar, parity, p.timeout_ns, p.status);
}

// all lanes wait, result made warp-uniform
__device__ __forceinline__ bool wait_warp(Ctl &c, uint32_t bar, uint32_t parity,
                                          const AttnParams &p) {
    return __all_sync(kFull, wait1(c, bar, parity, p));
}

template <int MODE>
__device__ __forceinline__ WorkItem fetch_item(const AttnParams &p, int w) {
    constexpr bool DENSE = MODE == kModeDense;
    WorkItem it{};
    if (w >= p.total_items) return it;
    const int uidx = w / p.pairs;
    const int pair = w - uidx * p.pairs;
    int unit = __ldg(p.sched + uidx);
    if (unit < 0 || unit >= p.U) {
        set_status(p.status, SIFT_ERR_DEVICE_CHECK);
        unit = uidx;
    }
    it.h = unit / p.N;
    it.i = unit - it.h * p.N;
    it.hq0 = it.h * p.G + 2 * pair;
    int n = __ldg(p.counts + unit);
    const int nmax = DENSE ? it.i + 1 : p.rowcap;
    if (n < 1 || n > nmax) {
        set_status(p.status, SIFT_ERR_DEVICE_CHECK);
        n = n < 1 ? 1 : nmax;
    }
    it.n = n;
    it.first = it.i - n + 1;
    it.list = (static_cast<int64_t>(it.h) * p.N + it.i) * p.rowcap;
    if constexpr (MODE == kModeRagged) {
        it.q0 = __ldg(p.qt + 2 * it.i);
        it.qlen = __ldg(p.qt + 2 * it.i + 1);
        if (it.q0 < 0 || it.qlen < 0 || it.qlen > p.B || it.q0 > p.total_tokens - it.qlen) {
            set_status(p.status, SIFT_ERR_DEVICE_CHECK);
            it.q0 = 0;
            it.qlen = 0;  // computed, never stored
        }
    }
    it.valid = 1;
    return it;
}

// entry j of the item's key-tile list (0 when j is past the end); bad sparse entries are
// reported and replaced by the diagonal tile so that every load stays inside the prompt
template <int MODE>
__device__ __forceinline__ int list_entry(const AttnParams &p, const WorkItem &it, int j) {
    constexpr bool DENSE = MODE == kModeDense;
    if (j >= it.n) return 0;
    if (DENSE) return it.first + j;
    int idx = __ldg(p.kv_idx + it.list + j);
    if (idx < 0 || idx > it.i || (j == it.n - 1 && idx != it.i)) {
        set_status(p.status, SIFT_ERR_DEVICE_CHECK);
        idx = it.i;
    }
    return idx;
}

// general layout: entry j of the item's list as (first, info); a gathered entry's first
// field is an index into the layer's page array.  Bad entries are reported and replaced
// by the item's own tile.
__device__ __forceinline__ int2 ragged_entry(const AttnParams &p, const WorkItem &it, int j) {
    if (j >= it.n) return make_int2(0, 0);
    int2 e = __ldg(&p.kv2[it.list + j]);
    const uint32_t info = static_cast<uint32_t>(e.y);
    bool ok;
    if (info & kGatherBit) {
        const int len = static_cast<int>(info & 0xffu);
        const int np = len / p.page;
        ok = j != it.n - 1 && len % p.page == 0 && np >= 1 && np * p.page <= p.B && e.x >= 0 &&
             e.x <= p.pages_len - np;
    } else {
        ok = e.x >= 0 && e.x <= it.q0 && (j != it.n - 1 || e.x == it.q0);
    }
    if (!ok) {
        set_status(p.status, SIFT_ERR_DEVICE_CHECK);
        e = make_int2(it.q0, 0);
    }
    return e;
}

// ---- rows walked from the bits ------------------------------------------------------
// Work order without a decode pass: by decreasing position inside the prompt (a row's
// tile count grows with its position), over prompts sorted by decreasing length, then
// kv head and head pair.  The CTA sorts the prompts once (Ctl::pord / plen).

// CA pages of documents g0+32*chunk .. : lane k loads document g0+32*chunk+k's start,
// tile count and first CA word (T = 0 for a document outside the range or malformed)
struct CaLane {
    int ds, T;
    int64_t off;
    uint64_t w0;
};

__device__ __forceinline__ CaLane ca_lane(const AttnParams &p, int p0, int g0, int g, int gk,
                                          int h) {
    CaLane r{0, 0, 0, 0};
    if (gk >= g) return r;
    r.ds = (gk == g0) ? p0 : __ldg(p.doc_end + gk - 1);
    const int de = __ldg(p.doc_end + gk);
    const int T = (de - r.ds) / p.B;
    const int W = (T + 63) / 64;
    r.off = __ldg(p.ca_off + gk) + (static_cast<int64_t>(p.layer) * p.Hkv + h) * W;
    if (de <= r.ds || (de - r.ds) % p.B || r.ds % p.B || r.off < 0 || r.off + W > p.ca_len) {
        set_status(p.status, SIFT_ERR_DEVICE_CHECK);
        return CaLane{0, 0, 0, 0};
    }
    r.T = T;
    r.w0 = __ldg(p.ca + r.off);
    return r;
}

__device__ __forceinline__ uint64_t low_bits(uint64_t word, int nb) {
    return nb >= 64 ? word : (nb <= 0 ? 0ull : (word & ((1ull << nb) - 1ull)));
}

// warp-collective: the item for work index w, with its tile count taken from the bits
__device__ WorkItem fetch_item_bits(const AttnParams &p, const Ctl &c, int w, uint32_t lane) {
    WorkItem it{};
    if (w >= p.total_items) return it;
    const int HP = p.Hkv * p.pairs;
    int64_t base = 0;
    int x = 0, rank = 0, rest = 0;
    bool found = false;
    for (int sgm = 0; sgm < p.P && !found; ++sgm) {
        const int lo = sgm + 1 < p.P ? c.plen[sgm + 1] : 0;
        const int64_t per = static_cast<int64_t>(sgm + 1) * HP;  // items per position
        const int64_t cnt = static_cast<int64_t>(c.plen[sgm] - lo) * per;
        if (w < base + cnt) {
            const int64_t off = w - base;
            x = c.plen[sgm] - 1 - static_cast<int>(off / per);
            const int r = static_cast<int>(off % per);
            rank = r / HP;
            rest = r % HP;
            found = true;
        }
        base += cnt;
    }
    if (!found) return it;  // the prompt lengths do not add up: nothing to do
    const int pr = c.pord[rank];
    it.h = rest / p.pairs;
    const int pair = rest % p.pairs;
    it.hq0 = it.h * p.G + 2 * pair;
    const int B = p.B;
    const int p0 = __ldg(p.cu + pr);
    it.pt = p0 / B;
    it.i = it.pt + x;
    it.g0 = __ldg(p.doc_cu + pr);
    int g1 = __ldg(p.doc_cu + pr + 1);
    if (it.g0 < 0 || it.g0 > g1 || g1 > p.D) {  // malformed: treat the prompt as all suffix
        set_status(p.status, SIFT_ERR_DEVICE_CHECK);
        it.g0 = g1 = 0;
    }
    // document of tile i: the first one ending after it (none: the query suffix)
    int lo = it.g0, hi = g1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.doc_end + mid) > it.i * B) hi = mid; else lo = mid + 1;
    }
    it.valid = 1;
    if (lo == g1) {
        it.g = -1;
        it.n = x + 1;
        return it;
    }
    it.g = lo;
    const int ds = (lo == it.g0) ? p0 : __ldg(p.doc_end + lo - 1);
    const int de = __ldg(p.doc_end + lo);
    const int T = (de - ds) / B;
    it.W = (T + 63) / 64;
    it.t0 = ds / B;
    const int il = it.i - it.t0;
    it.la_row = __ldg(p.la_off + lo) +
                ((static_cast<int64_t>(p.layer) * p.Hkv + it.h) * T + il) * it.W;
    int n = 1;  // the diagonal
    for (int b0 = it.g0; b0 < it.g; b0 += 32) {
        const CaLane cl = ca_lane(p, p0, it.g0, it.g, b0 + static_cast<int>(lane), it.h);
        int cnt = 0;
        const int Wk = (cl.T + 63) / 64;
        for (int wi = 0; wi < Wk; ++wi)
            cnt += __popcll(low_bits(wi == 0 ? cl.w0 : __ldg(p.ca + cl.off + wi), cl.T - 64 * wi));
        n += __reduce_add_sync(kFull, cnt);
    }
    if (de <= ds || (de - ds) % B || ds % B || it.la_row < 0 ||
        it.la_row + it.W > p.la_len) {
        set_status(p.status, SIFT_ERR_DEVICE_CHECK);
        it.W = 0;  // no LA words
    }
    int cnt = 0;
    for (int wi = static_cast<int>(lane); wi < it.W && 64 * wi < il; wi += 32)
        cnt += __popcll(low_bits(__ldg(p.la + it.la_row + wi), il - 64 * wi));
    n += __reduce_add_sync(kFull, cnt);
    it.n = min(n, p.rowcap);
    return it;
}

// warp-collective: visit(j) for every key tile of the item in ascending order -- CA pages
// of the earlier documents, LA tiles below the diagonal, the diagonal -- exactly it.n
// times; returns false as soon as visit does
template <typename F>
__device__ bool walk_bits(const AttnParams &p, const WorkItem &it, uint32_t lane, F &&visit) {
    if (it.g < 0) {
        for (int j = it.pt; j <= it.i; ++j)
            if (!visit(j)) return false;
        return true;
    }
    int done = 0;
    const int limit = it.n - 1;  // tiles before the diagonal
    const int p0 = it.pt * p.B;
    for (int b0 = it.g0; b0 < it.g && done < limit; b0 += 32) {
        const CaLane cl = ca_lane(p, p0, it.g0, it.g, b0 + static_cast<int>(lane), it.h);
        const int nd = min(32, it.g - b0);
        for (int k = 0; k < nd && done < limit; ++k) {
            const int Tq = __shfl_sync(kFull, cl.T, k);
            const int dsq = __shfl_sync(kFull, cl.ds, k);
            const int64_t offq = __shfl_sync(kFull, cl.off, k);
            const uint64_t wq = __shfl_sync(kFull, cl.w0, k);
            const int Wq = (Tq + 63) / 64;
            for (int wi = 0; wi < Wq && done < limit; ++wi) {
                uint64_t word = low_bits(wi == 0 ? wq : __ldg(p.ca + offq + wi), Tq - 64 * wi);
                while (word && done < limit) {
                    const int b = __ffsll(static_cast<long long>(word)) - 1;
                    word &= word - 1;
                    ++done;
                    if (!visit(dsq / p.B + 64 * wi + b)) return false;
                }
            }
        }
    }
    const int il = it.i - it.t0;
    for (int wi = 0; wi < it.W && 64 * wi < il && done < limit; ++wi) {
        uint64_t word = low_bits(__ldg(p.la + it.la_row + wi), il - 64 * wi);
        while (word && done < limit) {
            const int b = __ffsll(static_cast<long long>(word)) - 1;
            word &= word - 1;
            ++done;
            if (!visit(it.t0 + 64 * wi + b)) return false;
        }
    }
    for (; done < limit; ++done)  // only on malformed input (reported at fetch time)
        if (!visit(it.i)) return false;
    return visit(it.i);
}

// Columns c >= lim of a key tile are cleared (to -inf) in its first NW 32-column words (the
// words after them hide every column of the warp's rows and are not read): a word wholly
// below lim is left alone, the others compare column by column.
template <int BT, int NW>
__device__ __forceinline__ void mask_from(float (&x)[BT], int lim) {
#pragma unroll
    for (int w = 0; w < BT / 32 && w < NW; ++w) {
        const int c0 = 32 * w;
        if (lim < c0 + 32) {
#pragma unroll
            for (int t = 0; t < 32; ++t) x[c0 + t] = c0 + t < lim ? x[c0 + t] : -INFINITY;
        }
    }
}

// General layout: clear (to -inf) the columns of a key tile that row `row` may not use.
// info = len | causal << 8 | mask << 16: columns c < len whose page bit c >> lp is set,
// and c <= row on the diagonal.  When every page under the first len columns is kept
// (diagonal tiles, a partial last group of gathered pages, a partial last page) the
// visible columns are a prefix and one limit per row describes them; otherwise one
// 32-column visibility word at a time, words that are wholly visible skipping the selects.
__device__ __forceinline__ uint32_t page_word(uint32_t pm, int w, int lp) {
    if (lp >= 5) return ((pm >> ((32 * w) >> lp)) & 1u) ? kFull : 0u;  // one page per word
    if (lp == 4) {  // 2 pages of 16 columns: bit k -> bits [16k, 16k+16)
        const uint32_t b = (pm >> (2 * w)) & 0x3u;
        return ((b * 0x8001u) & 0x10001u) * 0xffffu;
    }
    if (lp == 3) {  // 4 pages of 8 columns: bit k -> byte k
        const uint32_t b = (pm >> (4 * w)) & 0xfu;
        return ((b * 0x00204081u) & 0x01010101u) * 0xffu;
    }
    uint32_t out = 0u;  // lp == 2: 8 pages of 4 columns (64-token tiles only)
    const uint32_t b = (pm >> (8 * w)) & 0xffu;
    for (int k = 0; k < 8; ++k)
        if ((b >> k) & 1u) out |= 0xfu << (4 * k);
    return out;
}

// the row's visible columns as one limit (columns c < limit), or -1 when a page under the
// first len columns is not kept
template <int BT>
__device__ __forceinline__ int prefix_limit(uint32_t info, int row, int lp) {
    const int len = static_cast<int>(info & 0xffu);
    const bool causal = (info >> 8) & 1u;
    const uint32_t pm = info >> 16;
    const int np = min((len + (1 << lp) - 1) >> lp, BT >> lp);  // pages under [0, len)
    const uint32_t need = (1u << np) - 1u;
    if ((pm & need) != need) return -1;
    return causal ? min(len, row + 1) : len;
}

// the visibility words of a tile whose kept pages leave holes
template <int BT>
__device__ __forceinline__ void mask_columns(float (&x)[BT], uint32_t info, int row, int lp) {
    const int len = static_cast<int>(info & 0xffu);
    const bool causal = (info >> 8) & 1u;
    const uint32_t pm = info >> 16;
#pragma unroll
    for (int w = 0; w < BT / 32; ++w) {
        const int c0 = 32 * w;
        uint32_t vis = len >= c0 + 32 ? kFull : (len <= c0 ? 0u : (1u << (len - c0)) - 1u);
        vis &= page_word(pm, w, lp);
        if (causal) vis &= row >= c0 + 31 ? kFull : (row < c0 ? 0u : (2u << (row - c0)) - 1u);
        if (vis != kFull) {
#pragma unroll
            for (int t = 0; t < 32; ++t)
                if (!((vis >> t) & 1u)) x[c0 + t] = -INFINITY;
        }
    }
}

template <int BT, int HD, int MODE>
__global__ void __launch_bounds__(threads_for(MODE != kModeRagged), 1)
sift_attention_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmKp,  // page-high boxes (gather)
                      const __grid_constant__ CUtensorMap tmVp,
                      const __grid_constant__ CUtensorMap tmO,  // O, tile-high boxes (stores)
                      const AttnParams p) {
    // whole tiles go out through a shared-memory staging tile and TMA stores, except on the
    // general layout (rows written by their softmax threads)
    constexpr bool STAGED = MODE != kModeRagged;
    using G = Geo<BT, HD, STAGED>;
    constexpr int kKSlots = G::kKSlots;
    constexpr bool DENSE = MODE == kModeDense;
    constexpr bool RAGGED = MODE == kModeRagged;  // list entries are first tokens, not tiles
    (void)DENSE;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    const uint32_t q_s = sbase;
    const uint32_t k_s = sbase + G::kKOff;
    const uint32_t v_s = sbase + G::kVOff;
    const uint32_t o_s = sbase + G::kOOff;
    Ctl &c = *reinterpret_cast<Ctl *>(smem + G::kCtlOff);

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31u;

    auto B_ = [&](const uint64_t &b) { return ptx::smem_u32(&b); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(B_(c.q_full[s]), 1);
            ptx::mbar_init(B_(c.q_empty[s]), 1);
        }
        for (int s = 0; s < kKSlots; ++s) {
            ptx::mbar_init(B_(c.k_full[s]), 1);
            ptx::mbar_init(B_(c.k_empty[s]), 1);
        }
        for (int s = 0; s < kVSlots; ++s) {
            ptx::mbar_init(B_(c.v_full[s]), 1);
            ptx::mbar_init(B_(c.v_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(B_(c.s_full[s]), 1);
            ptx::mbar_init(B_(c.p_half[s]), G::kSoftWarps);
            ptx::mbar_init(B_(c.p_full[s]), G::kSoftWarps);
            ptx::mbar_init(B_(c.o_full[s]), 1);
            ptx::mbar_init(B_(c.sch_full[s]), 1);
            // V producer, MMA issuer, the O writer (when staged), softmax warps of both heads
            ptx::mbar_init(B_(c.sch_empty[s]), (STAGED ? 3 : 2) + 2 * G::kSoftWarps);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(B_(c.stage_full[s]), G::kSoftWarps);
            ptx::mbar_init(B_(c.stage_free[s]), 1);
        }
        ptx::mbar_init(B_(c.teardown), 1);
        for (int r = 0; r < kRing; ++r) ptx::mbar_init(B_(c.ring_full[r]), 1);
        ptx::mbar_init(B_(c.never), 1);
        c.abort = 0;
        if (MODE == kModeBits) {
            // prompts by decreasing tile count (insertion sort; at most 64 prompts)
            for (int q = 0; q < p.P; ++q) {
                const int len = (__ldg(p.cu + q + 1) - __ldg(p.cu + q)) / p.B;
                int r = q;
                while (r > 0 && c.plen[r - 1] < len) {
                    c.plen[r] = c.plen[r - 1];
                    c.pord[r] = c.pord[r - 1];
                    --r;
                }
                c.plen[r] = len < 0 ? 0 : len;
                c.pord[r] = q;
            }
        }
        ptx::fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmO);
        if (RAGGED) {
            ptx::prefetch_tmap(&tmKp);
            ptx::prefetch_tmap(&tmVp);
        }
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(&c.tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = c.tmem_base;

    if (warp == kProducerWarp) {
        // ------------------------------------------------ scheduler + Q/K producer
        int item_k = 0, kf = 0;
        bool alive = true;
        const uint64_t pol_kv = ptx::policy_evict_last();   // K/V tiles are re-read by many items
        int w0 = 0;
        if (lane == 0) w0 = atomicAdd(p.work_counter, 1);
        auto fetch = [&](int w) {
            if constexpr (MODE == kModeBits) return fetch_item_bits(p, c, w, lane);
            else return fetch_item<MODE>(p, w);
        };
        WorkItem nxt = fetch(__shfl_sync(kFull, w0, 0));
        while (alive) {
            const WorkItem it = nxt;
            const int slot = item_k & 1;
            if (!wait_warp(c, B_(c.sch_empty[slot]), ((item_k >> 1) & 1) ^ 1, p)) break;
            if (lane == 0) {
                c.items[slot] = it;
                ptx::mbar_arrive(B_(c.sch_full[slot]));
            }
            __syncwarp();
            ++item_k;
            if (!it.valid) break;
            // claim the following item now, so that its tiles are known before this one
            // ends.  On decoded lists and dense rows longer than the K ring, its schedule
            // entry and count (dependent loads) are read only once this item's first K
            // tiles fill the ring, where they no longer hold back its first tile (aligned
            // 1-2% faster).  Elsewhere they are read at once: after a short row the next
            // item would wait for them, and on the general layout and on rows walked from
            // the bits the late read measured 1-7% slower.  (The next item's Q is not
            // pulled into L2 ahead: with a whole item of K/V passing through L2 in between,
            // 3% of the DRAM reads were such Q lines read twice.)
            int w = 0;
            if (lane == 0) w = atomicAdd(p.work_counter, 1);
            w = __shfl_sync(kFull, w, 0);
            constexpr bool kLateFetch = MODE == kModeList || MODE == kModeDense;
            bool fetched = !(kLateFetch && it.n > kKSlots);
            if (fetched) nxt = fetch(w);
            int k_in_item = 0;
            auto after_k = [&](bool ok) -> bool {
                if (ok && !fetched && ++k_in_item == kKSlots) {
                    nxt = fetch(w);
                    fetched = true;
                }
                return ok;
            };
            auto load_k = [&](int idx) -> bool {
                const int ks = kf % kKSlots;
                if (!wait_warp(c, B_(c.k_empty[ks]), ((kf / kKSlots) & 1) ^ 1, p)) return false;
                // lane 0 registers the bytes, then each box is issued by its own lane (a
                // thread issues bulk tensor copies slowly one after another)
                if (lane == 0) ptx::mbar_arrive_expect_tx(B_(c.k_full[ks]), G::kTxKV);
                __syncwarp();
                if (static_cast<int>(lane) < G::kBoxes)
                    ptx::tma_load_3d_hint(k_s + ks * G::kKVBytes + lane * G::kKVBox, &tmK,
                                          B_(c.k_full[ks]), 64 * lane, it.h,
                                          RAGGED ? idx : idx * BT, pol_kv);
                ++kf;
                return true;
            };
            // gathered pages: one page-high box per page into consecutive slots of the ring
            // slot (unused slots take the group's first page again, masked out later)
            auto load_k_pages = [&](int first, uint32_t info) -> bool {
                const int np = static_cast<int>(info & 0xffu) / p.page;
                int ps = 0;
                if (static_cast<int>(lane) < np) {
                    ps = __ldg(p.pages + first + lane);
                    if (ps < 0 || ps > it.q0) {
                        set_status(p.status, SIFT_ERR_DEVICE_CHECK);
                        ps = it.q0;
                    }
                }
                const int ks = kf % kKSlots;
                if (!wait_warp(c, B_(c.k_empty[ks]), ((kf / kKSlots) & 1) ^ 1, p)) return false;
                if (lane == 0) ptx::mbar_arrive_expect_tx(B_(c.k_full[ks]), G::kTxKV);
                __syncwarp();
                // one box per lane: lane = slot * boxes + box (at most 16 slots x 2 boxes)
                const int per = BT / p.page;
                const int sl = static_cast<int>(lane) / G::kBoxes, b = static_cast<int>(lane) % G::kBoxes;
                const int pst = __shfl_sync(kFull, ps, sl < np ? sl : 0);
                if (sl < per)
                    ptx::tma_load_3d_hint(k_s + ks * G::kKVBytes + b * G::kKVBox + sl * p.page * 128,
                                          &tmKp, B_(c.k_full[ks]), 64 * b, it.h, pst, pol_kv);
                ++kf;
                return true;
            };
            if constexpr (MODE == kModeBits) {
                alive = walk_bits(p, it, lane, [&](int idx) -> bool {
                    if (lane == 0) {  // published before the load, for the V producer
                        c.ring[kf % kRing] = idx;
                        ptx::mbar_arrive(B_(c.ring_full[kf % kRing]));
                    }
                    return load_k(idx);
                });
            } else if constexpr (RAGGED) {
                for (int jb = 0; jb < it.n && alive; jb += 32) {
                    const int2 e = ragged_entry(p, it, jb + static_cast<int>(lane));
                    const int cnt = min(32, it.n - jb);
                    for (int jj = 0; jj < cnt && alive; ++jj) {
                        const int x = __shfl_sync(kFull, e.x, jj);
                        const uint32_t info = __shfl_sync(kFull, static_cast<uint32_t>(e.y), jj);
                        alive = (info & kGatherBit) ? load_k_pages(x, info) : load_k(x);
                    }
                }
            } else {
                for (int jb = 0; jb < it.n && alive; jb += 32) {
                    const int idx_l = list_entry<MODE>(p, it, jb + static_cast<int>(lane));
                    const int cnt = min(32, it.n - jb);
                    for (int jj = 0; jj < cnt && alive; ++jj)
                        alive = after_k(load_k(__shfl_sync(kFull, idx_l, jj)));
                }
            }
            if (!fetched) nxt = fetch(w);
        }
        if (c.abort && lane == 0) {
            // unwinding: let every copy already issued land before shared memory is released
            for (int s = 0; s < kKSlots && s < kf; ++s) {
                const int last = s + ((kf - 1 - s) / kKSlots) * kKSlots;  // last fill of slot s
                drain_bar(B_(c.k_full[s]), (last / kKSlots) & 1, p.timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == kVProducerWarp) {
        // ------------------------------------------------ Q + V producer (runs behind the K producer)
        int item_k = 0, vf = 0, qk = 0;
        int q_issued[2] = {0, 0};  // Q loads issued per head slot (drained on abort)
        bool alive = true;
        const uint64_t pol_kv = ptx::policy_evict_last();
        const uint64_t pol_q = ptx::policy_evict_first();   // Q is read once per item
        while (alive) {
            const int slot = item_k & 1;
            if (!wait_warp(c, B_(c.sch_full[slot]), (item_k >> 1) & 1, p)) break;
            const WorkItem it = c.items[slot];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(B_(c.sch_empty[slot]));
            ++item_k;
            if (!it.valid) break;
            bool q_ok = true;
            for (int s = 0; s < 2 && q_ok; ++s) {
                if (!wait_warp(c, B_(c.q_empty[s]), (qk & 1) ^ 1, p)) {
                    q_ok = false;
                    break;
                }
                if (lane == 0) ptx::mbar_arrive_expect_tx(B_(c.q_full[s]), G::kTxQ / 2);
                __syncwarp();
                if (static_cast<int>(lane) < G::kBoxes)
                    ptx::tma_load_3d_hint(q_s + (s * G::kBoxes + lane) * G::kQBox, &tmQ,
                                          B_(c.q_full[s]), 64 * lane, it.hq0 + s,
                                          RAGGED ? it.q0 : it.i * BT, pol_q);
                ++q_issued[s];
            }
            if (!q_ok) break;
            ++qk;
            auto load_v = [&](int idx) -> bool {
                const int vs = vf % kVSlots;
                if (!wait_warp(c, B_(c.v_empty[vs]), ((vf / kVSlots) & 1) ^ 1, p)) return false;
                if (lane == 0) ptx::mbar_arrive_expect_tx(B_(c.v_full[vs]), G::kTxKV);
                __syncwarp();
                if (static_cast<int>(lane) < G::kBoxes)
                    ptx::tma_load_3d_hint(v_s + vs * G::kKVBytes + lane * G::kKVBox, &tmV,
                                          B_(c.v_full[vs]), 64 * lane, it.h,
                                          RAGGED ? idx : idx * BT, pol_kv);
                ++vf;
                return true;
            };
            auto load_v_pages = [&](int first, uint32_t info) -> bool {
                const int np = static_cast<int>(info & 0xffu) / p.page;
                int ps = 0;
                if (static_cast<int>(lane) < np) {
                    ps = __ldg(p.pages + first + lane);
                    if (ps < 0 || ps > it.q0) ps = it.q0;  // reported by the K producer
                }
                const int vs = vf % kVSlots;
                if (!wait_warp(c, B_(c.v_empty[vs]), ((vf / kVSlots) & 1) ^ 1, p)) return false;
                if (lane == 0) ptx::mbar_arrive_expect_tx(B_(c.v_full[vs]), G::kTxKV);
                __syncwarp();
                const int per = BT / p.page;
                const int sl = static_cast<int>(lane) / G::kBoxes, b = static_cast<int>(lane) % G::kBoxes;
                const int pst = __shfl_sync(kFull, ps, sl < np ? sl : 0);
                if (sl < per)
                    ptx::tma_load_3d_hint(v_s + vs * G::kKVBytes + b * G::kKVBox + sl * p.page * 128,
                                          &tmVp, B_(c.v_full[vs]), 64 * b, it.h, pst, pol_kv);
                ++vf;
                return true;
            };
            if constexpr (MODE == kModeBits) {
                // the K producer's tiles, in the same order (it walked the bits once)
                for (int j = 0; j < it.n && alive; ++j) {
                    const int r = vf % kRing;
                    if (!wait_warp(c, B_(c.ring_full[r]), (vf / kRing) & 1, p)) {
                        alive = false;
                        break;
                    }
                    alive = load_v(c.ring[r]);
                }
            } else if constexpr (RAGGED) {
                for (int jb = 0; jb < it.n && alive; jb += 32) {
                    const int2 e = ragged_entry(p, it, jb + static_cast<int>(lane));
                    const int cnt = min(32, it.n - jb);
                    for (int jj = 0; jj < cnt && alive; ++jj) {
                        const int x = __shfl_sync(kFull, e.x, jj);
                        const uint32_t info = __shfl_sync(kFull, static_cast<uint32_t>(e.y), jj);
                        alive = (info & kGatherBit) ? load_v_pages(x, info) : load_v(x);
                    }
                }
            } else {
                for (int jb = 0; jb < it.n && alive; jb += 32) {
                    const int idx_l = list_entry<MODE>(p, it, jb + static_cast<int>(lane));
                    const int cnt = min(32, it.n - jb);
                    for (int jj = 0; jj < cnt && alive; ++jj)
                        alive = load_v(__shfl_sync(kFull, idx_l, jj));
                }
            }
        }
        if (c.abort && lane == 0) {
            for (int s = 0; s < kVSlots && s < vf; ++s) {
                const int last = s + ((vf - 1 - s) / kVSlots) * kVSlots;
                drain_bar(B_(c.v_full[s]), (last / kVSlots) & 1, p.timeout_ns);
            }
            for (int s = 0; s < 2; ++s)
                if (q_issued[s] > 0) drain_bar(B_(c.q_full[s]), (q_issued[s] - 1) & 1, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer warp
        // Both heads' MMAs are issued in the order S0(j) | PV1(j-1) S1(j) |
        // PV0(j) S0(j+1) | ...: the heads alternate on the tensor pipe, each one's softmax
        // running while the other head's MMAs execute.
        {
            // The whole warp runs the issue loop on warp-uniform values (ring positions,
            // descriptors, waits made uniform by the vote) and one elected lane issues each
            // MMA and commit.  Run by a single lane, the loop lost about 7% end to end: its
            // operands first had to leave that lane's registers, on a sub-partition shared
            // with two busy softmax warps.
            if (p.stall) (void)wait_warp(c, B_(c.never), 0, p);
            int item_k = 0, qk = 0;
            // ring positions kept incrementally (no division on the issue path): K slot and
            // phase of the current tile, V slot and phase of the previous tile
            int ks = 0, vs = kVSlots - 1;
            uint32_t kph = 0, vph = 1;
            uint32_t pph0 = 0, pph1 = 0;
            const uint32_t tS0 = tmem, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
            // Descriptor bases.  The start address sits in the low 14 bits (16-byte units) and
            // every operand lies below 227 KB, so an in-bounds byte offset is added as
            // offset >> 4 without carrying into the other fields: one 64-bit add per MMA.
            const uint64_t dq = ptx::sdesc_sw128(q_s, 16, 1024);
            const uint64_t dk = ptx::sdesc_sw128(k_s, 16, 1024);
            const uint64_t dv = ptx::sdesc_sw128(v_s, G::kKVBox, 1024);
            auto commit = [&](uint32_t bar) {
                if (ptx::elect_one()) ptx::umma_commit(bar);
            };
            auto issue_s = [&](int s, int kslot) {
                const uint64_t qa = dq + static_cast<uint32_t>((s * G::kBoxes * G::kQBox) >> 4);
                const uint64_t kb = dk + static_cast<uint32_t>((kslot * G::kKVBytes) >> 4);
                const uint32_t d = s ? tS1 : tS0;
                if (ptx::elect_one()) ptx::umma_ss_c<false>(d, qa, kb, G::kIdescS);
#pragma unroll
                for (int kk = 1; kk < HD / 16; ++kk) {
                    const uint32_t off_q = ((kk >> 2) * G::kQBox + (kk & 3) * 32) >> 4;
                    const uint32_t off_k = ((kk >> 2) * G::kKVBox + (kk & 3) * 32) >> 4;
                    if (ptx::elect_one()) ptx::umma_ss_c<true>(d, qa + off_q, kb + off_k, G::kIdescS);
                }
            };
            // P*V of head s: the MMAs over the first half of the keys go out as soon as that
            // half of P is in tensor memory, while the softmax still works on the second
            auto issue_pv = [&](int s, int vslot, bool acc) -> bool {
                const uint64_t vb = dv + static_cast<uint32_t>((vslot * G::kKVBytes) >> 4);
                const uint32_t d = s ? tO1 : tO0;
                const uint32_t a = s ? tS1 : tS0;
                uint32_t &ph = s ? pph1 : pph0;
                if (!wait_warp(c, B_(c.p_half[s]), ph, p)) return false;
                ptx::tc_fence_after();
                if (ptx::elect_one()) {
                    if (acc) ptx::umma_ts_c<true>(d, a, vb, G::kIdescPV);
                    else ptx::umma_ts_c<false>(d, a, vb, G::kIdescPV);
                }
#pragma unroll
                for (int kk = 1; kk < BT / 32; ++kk)
                    if (ptx::elect_one())
                        ptx::umma_ts_c<true>(d, a + kk * 8, vb + ((kk * 16 * 128) >> 4), G::kIdescPV);
                if (!wait_warp(c, B_(c.p_full[s]), ph, p)) return false;
                ph ^= 1;
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = BT / 32; kk < BT / 16; ++kk)
                    if (ptx::elect_one())
                        ptx::umma_ts_c<true>(d, a + kk * 8, vb + ((kk * 16 * 128) >> 4), G::kIdescPV);
                return true;
            };
            // An item's last P*V pair (the "tail") completes its O; it goes out before the
            // next item's first S.  (Issuing each head's tail right before that head's next
            // S instead, across the item boundary, gained 1.7% on the general layout while
            // P was handed over whole; with P in halves it lost 1.2% there, 0.3% aligned.)
            bool ok = true;
            auto issue_tail = [&](int n_tiles) -> bool {
                if (!wait_warp(c, B_(c.v_full[vs]), vph, p) || !issue_pv(0, vs, n_tiles > 1))
                    return false;
                commit(B_(c.o_full[0]));
                if (!issue_pv(1, vs, n_tiles > 1)) return false;
                commit(B_(c.o_full[1]));
                return true;
            };
            while (__shfl_sync(kFull, c.abort, 0) == 0) {  // one read for the whole warp
                const int slot = item_k & 1;
                if (!wait_warp(c, B_(c.sch_full[slot]), (item_k >> 1) & 1, p)) { ok = false; break; }
                // the item's tile count, uniform across the warp
                const int valid = __shfl_sync(kFull, c.items[slot].valid, 0);
                const int n_tiles = __shfl_sync(kFull, c.items[slot].n, 0);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(B_(c.sch_empty[slot]));
                ++item_k;
                if (!valid) break;
                const uint32_t qph = qk & 1;
                ++qk;
                for (int j = 0; j < n_tiles; ++j) {
                    // this tile's K (and at its first tile, head 0's Q of the item)
                    if ((j == 0 && !wait_warp(c, B_(c.q_full[0]), qph, p)) ||
                        !wait_warp(c, B_(c.k_full[ks]), kph, p)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    // P*V of the previous tile (vs names its V)
                    if (j > 0 && (!wait_warp(c, B_(c.v_full[vs]), vph, p) || !issue_pv(0, vs, j > 1))) {
                        ok = false;
                        break;
                    }
                    issue_s(0, ks);
                    commit(B_(c.s_full[0]));
                    if (j > 0 && !issue_pv(1, vs, j > 1)) { ok = false; break; }
                    if (j == 0) {  // head 1's Q of this item
                        if (!wait_warp(c, B_(c.q_full[1]), qph, p)) { ok = false; break; }
                        ptx::tc_fence_after();
                    }
                    issue_s(1, ks);
                    commit(B_(c.s_full[1]));
                    // advance: this tile's V becomes "previous", the K ring moves on
                    if (++vs == kVSlots) { vs = 0; vph ^= 1; }
                    if (++ks == kKSlots) { ks = 0; kph ^= 1; }
                }
                if (!ok || !issue_tail(n_tiles)) break;
            }
            // every MMA issued so far must finish before TMEM and shared memory go away
            commit(B_(c.teardown));
            drain_bar(B_(c.teardown), 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp < kProducerWarp) {
        // ------------------------------------------------ softmax + epilogue
        const int s = warp >> 2;
        const int wq = warp & 3;
        if (wq < G::kSoftWarps) {
            const int row = wq * 32 + static_cast<int>(lane);
            const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
            const uint32_t tS = tmem + lane_off + s * 128;
            const uint32_t tO = tmem + lane_off + 256 + s * 128;
            const float sl2 = p.scale_log2;
            int item_k = 0;
            uint32_t sph = 0, oph = 0;
            // The first warp of head slot 1 hands buffers back to the producers: S1(j) is the
            // last MMA to read K_j and Q (at the item's last tile), and completes after
            // PV1(j-1), the last reader of V_{j-1}; o_full of slot 1 covers the item's last V.
            const bool releaser = (s == 1 && wq == 0 && lane == 0);
            // and the first warp of head slot 0 hands back that slot's Q after its last S
            const bool q0_releaser = (s == 0 && wq == 0 && lane == 0);
            int t = 0;  // key tiles seen so far, same order as the producers and the MMA issuer
            int n_staged = 0;  // this head's tiles written through the staging tile so far
            while (true) {
                const int slot = item_k & 1;
                if (!wait_warp(c, B_(c.sch_full[slot]), (item_k >> 1) & 1, p)) break;
                const WorkItem it = c.items[slot];
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(B_(c.sch_empty[slot]));
                ++item_k;
                if (!it.valid) break;
                float m = -INFINITY, l = 0.f;
                bool ok = true;
                for (int j = 0; j < it.n; ++j) {
                    uint32_t info = 0;  // general layout: this key tile's length / causal / pages
                    if constexpr (RAGGED) info = static_cast<uint32_t>(__ldg(&p.kv2[it.list + j].y));
                    (void)info;
                    if (!wait_warp(c, B_(c.s_full[s]), sph, p)) { ok = false; break; }
                    sph ^= 1;
                    if (releaser) {
                        ptx::mbar_arrive(B_(c.k_empty[t % kKSlots]));
                        if (j > 0) ptx::mbar_arrive(B_(c.v_empty[(t + kVSlots - 1) % kVSlots]));
                        if (j == it.n - 1) ptx::mbar_arrive(B_(c.q_empty[1]));
                    }
                    if (q0_releaser && j == it.n - 1) ptx::mbar_arrive(B_(c.q_empty[0]));
                    ++t;
                    ptx::tc_fence_after();
                    float x[BT];
                    if constexpr (BT == 128) ptx::tmem_ld128(tS, x); else ptx::tmem_ld64(tS, x);
                    // A tile whose visible columns are a prefix of each row (the diagonal; on
                    // the general layout also partial groups and pages) is masked by a limit
                    // per row.  On the diagonal, a warp whose rows all end in the first half
                    // of the keys (warp-uniform) runs a copy of the code without the second
                    // half: no max, no exponentials, P = 0 there.  (The general layout, whose
                    // masked tiles are frequent, keeps one copy: switching between two cost
                    // it 15% while the aligned layouts gained 1-4%.)
                    int lim = -1;
                    if constexpr (RAGGED) {
                        if ((info & ~kGatherBit) != p.full_info) {
                            lim = prefix_limit<BT>(info, row, p.lp);
                            // Pages whose kept bits leave holes in a tile come only from
                            // 4-token pages under 64-token tiles (larger pages below the
                            // tile are gathered, and pages of a tile or more are one bit).
                            // The 128-token kernel leaves that code out (2% on its general
                            // layout) and reports such an entry, read as its first len keys.
                            if constexpr (BT == 64) {
                                if (lim < 0) mask_columns<BT>(x, info, row, p.lp);
                            } else if (lim < 0) {
                                set_status(p.status, SIFT_ERR_DEVICE_CHECK);
                                lim = static_cast<int>(info & 0xffu);
                                if ((info >> 8) & 1u) lim = min(lim, row + 1);
                            }
                        }
                    } else if (j == it.n - 1) {
                        lim = row + 1;  // the diagonal tile: keys up to the row's own
                    }
                    int nw = BT / 32;  // leading 32-column words visible to some row of the warp
                    if (!RAGGED && lim >= 0)  // uniform: the diagonal tile, for the whole warp
                        nw = (__reduce_max_sync(kFull, static_cast<unsigned>(lim)) + 31) >> 5;
                    auto tile = [&](auto nw_c) {
                        constexpr int NW = decltype(nw_c)::value;
                        if (lim >= 0) mask_from<BT, NW>(x, lim);
                        // row max: independent three-input chains of 32 columns each
                        float mxc[BT / 32];
#pragma unroll
                        for (int q = 0; q < BT / 32; ++q) {
                            mxc[q] = -INFINITY;
                            if (q < NW) {
                                const float *xb = x + 32 * q;
                                float a = ptx::fmax3(xb[0], xb[1], xb[2]);
#pragma unroll
                                for (int t = 3; t < 31; t += 2) a = ptx::fmax3(a, xb[t], xb[t + 1]);
                                mxc[q] = fmaxf(a, xb[31]);
                            }
                        }
                        float mx = fmaxf(mxc[0], mxc[1]);
                        if constexpr (BT == 128) mx = ptx::fmax3(mx, mxc[2], mxc[3]);
                        const float m_new = fmaxf(m, mx * sl2);
                        const bool need = m_new > m + 8.0f;
                        float alpha = 1.f;
                        if (need) {
                            alpha = ptx::ex2(m - m_new);
                            m = m_new;
                        }
                        // p = 2^(x*scale*log2e - m): packed FMA, MUFU ex2, packed partial sums.
                        // Each half of the keys goes to the MMA issuer as soon as it is stored.
                        const uint64_t sl2x2 = ptx::f2(sl2, sl2);
                        const uint64_t nmb = ptx::f2(-m, -m);
                        uint64_t acc[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[q] = ptx::f2(0.f, 0.f);
                        uint32_t pk[BT / 2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
#pragma unroll
                            for (int t = h * (BT / 4); t < (h + 1) * (BT / 4); ++t) {
                                if (t < 16 * NW) {
                                    float e0, e1;
                                    ptx::f2_split(ptx::ffma2(ptx::f2(x[2 * t], x[2 * t + 1]), sl2x2, nmb),
                                                  e0, e1);
                                    const float p0 = ptx::ex2(e0), p1 = ptx::ex2(e1);
                                    acc[t & 3] = ptx::fadd2(acc[t & 3], ptx::f2(p0, p1));
                                    pk[t] = ptx::pack_bf16x2(p0, p1);
                                } else {
                                    pk[t] = 0u;
                                }
                            }
                            const uint32_t(&half)[BT / 4] =
                                *reinterpret_cast<const uint32_t(*)[BT / 4]>(pk + h * (BT / 4));
                            if constexpr (BT == 128) ptx::tmem_st32(tS + h * 32, half);
                            else ptx::tmem_st16(tS + h * 16, half);
                            // O takes the new max before any of this tile's P reaches the tensor
                            // pipe (this head's P*V of the previous tile finished before its S did)
                            if (h == 0 && j > 0 && __any_sync(kFull, need)) {
#pragma unroll 1
                                for (int cc = 0; cc < HD / 32; ++cc) {
                                    float ov[32];
                                    ptx::tmem_ld32(tO + cc * 32, ov);
#pragma unroll
                                    for (int t = 0; t < 32; ++t) ov[t] *= alpha;
                                    ptx::tmem_st32f(tO + cc * 32, ov);
                                }
                            }
                            ptx::tc_fence_before();
                            __syncwarp();
                            if (lane == 0) ptx::mbar_arrive(B_(h == 0 ? c.p_half[s] : c.p_full[s]));
                        }
                        float a0, a1;
                        ptx::f2_split(ptx::fadd2(ptx::fadd2(acc[0], acc[1]), ptx::fadd2(acc[2], acc[3])),
                                      a0, a1);
                        l = l * alpha + (a0 + a1);
                    };
                    if (!RAGGED && nw <= BT / 64) tile(std::integral_constant<int, BT / 64>{});
                    else tile(std::integral_constant<int, BT / 32>{});
                }
                if (!ok) break;
                if (!wait_warp(c, B_(c.o_full[s]), oph, p)) break;
                oph ^= 1;
                // the item's last V slot: head 1 stages its O there on staged layouts (the
                // O writer hands the slot back once the store has read it)
                const int last_vslot = (t + kVSlots - 1) % kVSlots;
                if (releaser && !STAGED) ptx::mbar_arrive(B_(c.v_empty[last_vslot]));
                ptx::tc_fence_after();
                // Aligned tiles are staged in shared memory and go out as one TMA store per
                // box; the general layout's tiles are written row by row (a partial one must
                // not spill into the next segment, and the stores would compete with its
                // gathered page loads).  Head 0 stages in the staging tile, once the store of
                // its previous tile has read it; head 1 in the slot of the item's last V tile,
                // free as soon as P*V is done (o_full).  (When both heads took the staging
                // tile in turn, head 1's epilogue waited for head 0's store: 2,970 cycles
                // against head 0's 1,120, which held back head 1's next softmax.)
                const bool staged = STAGED;
                if (staged && s == 0 && n_staged > 0 &&
                    !wait_warp(c, B_(c.stage_free[0]), (n_staged - 1) & 1, p))
                    break;
                const float inv = 1.f / l;
                const int64_t tok = RAGGED ? static_cast<int64_t>(it.q0) + row
                                           : static_cast<int64_t>(it.i) * BT + row;
                const int hq = it.hq0 + s;
                uint4 *orow = reinterpret_cast<uint4 *>(p.o + (tok * p.Hq + hq) * HD);
                // rows past the segment's end are not stored; every lane still takes part
                // in the warp-collective tensor-memory loads
                const bool store = !RAGGED || row < it.qlen;
                // this row in the staging tile: box cc/2, 128 bytes per row, 16-byte chunks
                // placed by the 128-byte swizzle (chunk k of row r at k ^ (r % 8))
                const uint32_t srow =
                    (s == 0 ? o_s : v_s + static_cast<uint32_t>(last_vslot) * G::kKVBytes) +
                    static_cast<uint32_t>(row) * 128u;
#pragma unroll 1
                for (int cc = 0; cc < HD / 32; ++cc) {
                    float ov[32];
                    ptx::tmem_ld32(tO + cc * 32, ov);
                    uint32_t pk[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        pk[t] = ptx::pack_bf16x2(ov[2 * t] * inv, ov[2 * t + 1] * inv);
                    if (staged) {
                        const uint32_t box = srow + static_cast<uint32_t>(cc >> 1) * G::kOBox;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t chunk = static_cast<uint32_t>((cc & 1) * 4 + k);
                            ptx::st_shared_v4(box + ((chunk ^ static_cast<uint32_t>(row & 7)) << 4),
                                              pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                        }
                    } else if (store) {
                        if (p.o_v8) {  // whole 32-byte sectors: half the store instructions
                            ptx::st_global_v8(orow + cc * 4, pk);
                            ptx::st_global_v8(orow + cc * 4 + 2, pk + 8);
                        } else {
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4)
                                orow[cc * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1],
                                                               pk[4 * v4 + 2], pk[4 * v4 + 3]);
                        }
                    }
                }
                if (staged) {
                    ptx::fence_proxy_async_smem();  // the TMA store reads what these threads wrote
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(B_(c.stage_full[s]));
                    ++n_staged;
                }
                if (store)
                    p.lse[static_cast<int64_t>(hq) * p.total_tokens + tok] =
                        (m + log2f(l)) * 0.69314718055994530942f;
                ptx::tc_fence_before();
            }
        }
    } else if (STAGED && warp == kStoreWarp) {
        // ------------------------------------------------ O writer
        // Follows the items; for each whole tile, head 0's then head 1's staged O goes out
        // as one TMA store per 64-column box (one lane per box).  Once a store has read its
        // tile, head 0's staging tile goes back to head 0 and head 1's (the item's last V
        // slot) to the V producer.
        int item_k = 0, n = 0, t = 0;
        bool issued = false;
        while (true) {
            const int slot = item_k & 1;
            if (!wait_warp(c, B_(c.sch_full[slot]), (item_k >> 1) & 1, p)) break;
            const WorkItem it = c.items[slot];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(B_(c.sch_empty[slot]));
            ++item_k;
            if (!it.valid) break;
            const int tok0 = RAGGED ? it.q0 : it.i * BT;
            t += it.n;
            const int last_vslot = (t + kVSlots - 1) % kVSlots;
            bool ok = true;
            for (int s = 0; s < 2; ++s) {
                if (!wait_warp(c, B_(c.stage_full[s]), n & 1, p)) {
                    ok = false;
                    break;
                }
                const uint32_t src =
                    s == 0 ? o_s : v_s + static_cast<uint32_t>(last_vslot) * G::kKVBytes;
                if (static_cast<int>(lane) < G::kBoxes) {
                    ptx::tma_store_3d(&tmO, src + lane * G::kOBox, 64 * lane, it.hq0 + s, tok0);
                    ptx::bulk_commit();
                    ptx::bulk_wait_read();
                    issued = true;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(B_(s == 0 ? c.stage_free[0] : c.v_empty[last_vslot]));
            }
            if (!ok) break;
            ++n;
        }
        // every store must have landed before the kernel ends
        if (issued) ptx::bulk_wait_all();
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// [tokens][heads][d] bf16 viewed as a 3-D tensor (d, heads, tokens); box 64 x 1 x rows
bool make_map(CUtensorMap *m, const void *base, int d, int heads, int tokens, int rows) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                          static_cast<cuuint64_t>(tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(heads) * d * 2};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int BT, int HD, int MODE>
sift_status launch_attention(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                             const CUtensorMap &mkp, const CUtensorMap &mvp, const CUtensorMap &mo,
                             const AttnParams &p, cudaStream_t stream) {
    using G = Geo<BT, HD, MODE != kModeRagged>;
    auto kern = sift_attention_kernel<BT, HD, MODE>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        G::kSmem);
    });
    if (attr_err != cudaSuccess) return SIFT_ERR_CUDA;
    const int sms = device_sm_count();
    if (sms <= 0) return SIFT_ERR_CUDA;
    const int grid = p.total_items < sms ? p.total_items : sms;
    if (grid <= 0) return SIFT_OK;
    kern<<<grid, threads_for(MODE != kModeRagged), G::kSmem, stream>>>(mq, mk, mv, mkp, mvp, mo, p);
    return cudaGetLastError() == cudaSuccess ? SIFT_OK : SIFT_ERR_CUDA;
}

// maps: Q, K, V with tile-high boxes, then K, V with page-high boxes (gathered pages of
// the general layout; the tile-high ones again everywhere else), then O with tile-high
// boxes (stores)
template <int MODE>
sift_status dispatch(int tile, int hd, const CUtensorMap *m, const AttnParams &p,
                     cudaStream_t stream) {
    if (tile == 128 && hd == 128)
        return launch_attention<128, 128, MODE>(m[0], m[1], m[2], m[3], m[4], m[5], p, stream);
    if (tile == 128 && hd == 64)
        return launch_attention<128, 64, MODE>(m[0], m[1], m[2], m[3], m[4], m[5], p, stream);
    if (tile == 64 && hd == 128)
        return launch_attention<64, 128, MODE>(m[0], m[1], m[2], m[3], m[4], m[5], p, stream);
    if (tile == 64 && hd == 64)
        return launch_attention<64, 64, MODE>(m[0], m[1], m[2], m[3], m[4], m[5], p, stream);
    return SIFT_ERR_UNSUPPORTED;
}

sift_status prepare(const sift_problem *prob, const void *q, const void *k, const void *v,
                    float softmax_scale, void *o, float *lse, void *workspace,
                    size_t workspace_bytes, int32_t *dev_status, CUtensorMap *maps,
                    AttnParams *p, int num_query_tiles = 0) {
    // num_query_tiles > 0: the general layout, whose query tiles are counted per segment
    sift_status st = num_query_tiles > 0 ? validate_ragged(prob, true) : validate_problem(prob, true);
    if (st != SIFT_OK) return st;
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || lse == nullptr ||
        workspace == nullptr || dev_status == nullptr)
        return SIFT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0)
        return SIFT_ERR_INVALID_ARG;
    if (workspace_bytes < sift_workspace_bytes(prob)) return SIFT_ERR_INVALID_ARG;
    const int d = prob->head_dim, B = prob->tile, T = prob->total_tokens;
    if (!make_map(&maps[0], q, d, prob->num_q_heads, T, B) ||
        !make_map(&maps[1], k, d, prob->num_kv_heads, T, B) ||
        !make_map(&maps[2], v, d, prob->num_kv_heads, T, B))
        return SIFT_ERR_CUDA;
    maps[3] = maps[1];
    maps[4] = maps[2];
    if (!make_map(&maps[5], o, d, prob->num_q_heads, T, B)) return SIFT_ERR_CUDA;
    const int N = num_query_tiles > 0 ? num_query_tiles : T / B;
    const int G = prob->num_q_heads / prob->num_kv_heads;
    AttnParams a{};
    a.o = static_cast<__nv_bfloat16 *>(o);
    a.o_v8 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
    a.lse = lse;
    a.work_counter = static_cast<int32_t *>(workspace);
    a.status = dev_status;
    a.U = N * prob->num_kv_heads;
    a.N = N;
    a.Hq = prob->num_q_heads;
    a.G = G;
    a.pairs = G / 2;
    const int64_t items = static_cast<int64_t>(a.U) * a.pairs;
    if (items > INT32_MAX / 2) return SIFT_ERR_UNSUPPORTED;
    a.total_items = static_cast<int32_t>(items);
    a.rowcap = prob->max_tiles_per_prompt;
    a.total_tokens = T;
    const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(d));
    a.scale_log2 = scale * 1.4426950408889634f;
    const DebugWaits dw = debug_waits();
    a.timeout_ns = dw.timeout_ns;
    a.stall = dw.stall;
    *p = a;
    return SIFT_OK;
}

}  // namespace
}  // namespace sift

extern "C" sift_status sift_sparse_prefill(const sift_problem *prob, int32_t layer, const void *q,
                                           const void *k, const void *v, const int32_t *kv_idx,
                                           const int32_t *counts, const int32_t *sched,
                                           float softmax_scale, void *o, float *lse,
                                           void *workspace, size_t workspace_bytes,
                                           int32_t *dev_status, cudaStream_t stream) {
    using namespace sift;
    NvtxRange nvtx_range("sift_sparse_prefill");
    if (prob == nullptr || layer < 0 || layer >= prob->num_layers || kv_idx == nullptr ||
        counts == nullptr || sched == nullptr)
        return SIFT_ERR_INVALID_ARG;
    CUtensorMap maps[6];
    AttnParams p;
    sift_status st = prepare(prob, q, k, v, softmax_scale, o, lse, workspace, workspace_bytes,
                             dev_status, maps, &p);
    if (st != SIFT_OK) return st;
    const int64_t lu = static_cast<int64_t>(layer) * p.U;
    p.kv_idx = kv_idx + lu * p.rowcap;
    p.counts = counts + lu;
    p.sched = sched + lu;
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), stream) != cudaSuccess) return SIFT_ERR_CUDA;
    return dispatch<kModeList>(prob->tile, prob->head_dim, maps, p, stream);
}

extern "C" sift_status sift_sparse_prefill_ragged(const sift_problem *prob, int32_t num_query_tiles,
                                                  int32_t layer, const void *q, const void *k,
                                                  const void *v, const int32_t *qtiles,
                                                  const int32_t *kv, const int32_t *counts,
                                                  const int32_t *sched, const int32_t *pages,
                                                  int32_t page_cap, float softmax_scale,
                                                  void *o, float *lse, void *workspace,
                                                  size_t workspace_bytes, int32_t *dev_status,
                                                  cudaStream_t stream) {
    using namespace sift;
    NvtxRange nvtx_range("sift_sparse_prefill_ragged");
    if (prob == nullptr || layer < 0 || layer >= prob->num_layers || qtiles == nullptr ||
        kv == nullptr || counts == nullptr || sched == nullptr || num_query_tiles < 1 ||
        (reinterpret_cast<uintptr_t>(kv) & 7u) != 0)
        return SIFT_ERR_INVALID_ARG;
    const bool gather = gathers_pages(prob) && prob->num_docs > 0;
    if (gather && (pages == nullptr || page_cap < 1 ||
                   static_cast<int64_t>(prob->num_kv_heads) * prob->num_docs * page_cap > INT32_MAX))
        return SIFT_ERR_INVALID_ARG;
    if (validate_ragged(prob, true) == SIFT_OK && num_query_tiles > max_query_tiles(prob))
        return SIFT_ERR_INVALID_ARG;
    CUtensorMap maps[6];
    AttnParams p;
    sift_status st = prepare(prob, q, k, v, softmax_scale, o, lse, workspace, workspace_bytes,
                             dev_status, maps, &p, num_query_tiles);
    if (st != SIFT_OK) return st;
    const int64_t lu = static_cast<int64_t>(layer) * p.U;
    p.kv2 = reinterpret_cast<const int2 *>(kv) + lu * p.rowcap;
    p.counts = counts + lu;
    p.sched = sched + lu;
    p.qt = qtiles;
    p.B = prob->tile;
    const int page = prob->page ? prob->page : prob->tile;
    p.page = page;
    if (gather) {
        const int64_t slice = static_cast<int64_t>(prob->num_kv_heads) * prob->num_docs * page_cap;
        p.pages = pages + layer * slice;
        p.pages_len = slice;
        // gathered pages land page rows at a time (slot offsets are multiples of 1024 bytes,
        // so the 128-byte swizzle phase of the tile is kept)
        if (!make_map(&maps[3], k, prob->head_dim, prob->num_kv_heads, prob->total_tokens, page) ||
            !make_map(&maps[4], v, prob->head_dim, prob->num_kv_heads, prob->total_tokens, page))
            return SIFT_ERR_CUDA;
    } else {
        p.pages = nullptr;
        p.pages_len = 0;
    }
    const int pin = page < prob->tile ? page : prob->tile;
    int lp = 0;
    while ((1 << lp) < pin) ++lp;
    p.lp = lp;
    p.full_info = static_cast<uint32_t>(prob->tile) |
                  ((1u << (prob->tile / pin)) - 1u) << 16;
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), stream) != cudaSuccess) return SIFT_ERR_CUDA;
    return dispatch<kModeRagged>(prob->tile, prob->head_dim, maps, p, stream);
}

extern "C" sift_status sift_dense_prefill(const sift_problem *prob, const void *q, const void *k,
                                          const void *v, float softmax_scale, void *o, float *lse,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t *dev_status, cudaStream_t stream) {
    using namespace sift;
    NvtxRange nvtx_range("sift_dense_prefill");
    CUtensorMap maps[6];
    AttnParams p;
    sift_status st = prepare(prob, q, k, v, softmax_scale, o, lse, workspace, workspace_bytes,
                             dev_status, maps, &p);
    if (st != SIFT_OK) return st;
    int32_t *ws_counts = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + kWsHeader);
    int32_t *ws_sched = ws_counts + p.U;
    if (launch_dense_counts(prob, ws_counts, dev_status, stream) != cudaSuccess)
        return SIFT_ERR_CUDA;
    if (launch_schedule(ws_counts, ws_sched, 1, p.U, prob->max_tiles_per_prompt, dev_status,
                        stream) != cudaSuccess)
        return SIFT_ERR_CUDA;
    p.kv_idx = nullptr;
    p.counts = ws_counts;
    p.sched = ws_sched;
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), stream) != cudaSuccess) return SIFT_ERR_CUDA;
    return dispatch<kModeDense>(prob->tile, prob->head_dim, maps, p, stream);
}

extern "C" sift_status sift_fused_prefill(const sift_problem *prob, int32_t layer,
                                          const uint64_t *la_words, const uint64_t *ca_words,
                                          const void *q, const void *k, const void *v,
                                          float softmax_scale, void *o, float *lse,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t *dev_status, cudaStream_t stream) {
    using namespace sift;
    NvtxRange nvtx_range("sift_fused_prefill");
    if (prob == nullptr || layer < 0 || layer >= prob->num_layers) return SIFT_ERR_INVALID_ARG;
    if ((prob->la_words_len > 0 && la_words == nullptr) ||
        (prob->ca_words_len > 0 && ca_words == nullptr))
        return SIFT_ERR_INVALID_ARG;
    if (prob->num_prompts > kMaxFusedPrompts) return SIFT_ERR_UNSUPPORTED;
    CUtensorMap maps[6];
    AttnParams p;
    sift_status st = prepare(prob, q, k, v, softmax_scale, o, lse, workspace, workspace_bytes,
                             dev_status, maps, &p);
    if (st != SIFT_OK) return st;
    p.kv_idx = nullptr;
    p.counts = nullptr;
    p.sched = nullptr;
    p.cu = prob->cu_seqlens;
    p.doc_cu = prob->doc_cu;
    p.doc_end = prob->doc_end;
    p.la_off = prob->la_off;
    p.ca_off = prob->ca_off;
    p.la = la_words;
    p.ca = ca_words;
    p.la_len = prob->la_words_len;
    p.ca_len = prob->ca_words_len;
    p.P = prob->num_prompts;
    p.D = prob->num_docs;
    p.B = prob->tile;
    p.layer = layer;
    p.Hkv = prob->num_kv_heads;
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), stream) != cudaSuccess) return SIFT_ERR_CUDA;
    return dispatch<kModeBits>(prob->tile, prob->head_dim, maps, p, stream);
}
