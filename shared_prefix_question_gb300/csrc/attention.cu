// attention.cu -- prefix-tail attention on tcgen05 tensor cores (blink.py PREFIX_CACHE note and
// `_forward_shared`: every tail runs against the one shared prefix KV, same tokens and positions).
//
// Work decomposition.  Rows of the M dimension are (tail token, query head of one GQA group):
// a 128-row tile holds tpt = 128 / g consecutive tokens times the g query heads that share one
// kv head, so every K/V tile staged in shared memory serves all g heads.  A thread block owns
// two such tiles (256 rows) of one kv head and sweeps the KV sequence:
//   - the prefix tiles (all P prefix keys, no mask: every tail row sees every prefix key), then
//   - the tail tiles: keys from the first question touched by the block up to its last token,
//     masked per row to its own question (key >= question start) and causally (key <= token).
// The running (max, sum) online softmax merges the parts: each new KV tile is folded into the
// accumulator by log-sum-exp rescaling, which is exactly the LSE merge of the prefix and tail
// partial results.
//
// Roles (320 threads):
//   warp 8       TMA producer: Q tiles once, then K/V tiles into a ring of 4 shared-memory slots;
//   warp 9       MMA issuer (one thread): S_t = Q_t K^T into tensor memory, O_t += P_t V with P_t
//                read straight from tensor memory;
//   warps 0-3/4-7 softmax for tile 0 / tile 1, one row per thread: reads S from tensor memory,
//                masks, keeps (m, l), writes P (bf16) over S, rescales O lazily (only when the
//                row max grew by more than 2^8), and finally normalises O and stores it.
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// MMA issue order: S0(i), PV1(i-1), S1(i), PV0(i), so each softmax warpgroup works while the
// tensor core runs the other tile's products.
//
// Small grids (one request whose blocks fill at most half of the SMs, e.g. one question against
// a long prefix) and the last partial wave of a launch: the prefix tiles of some units are cut
// into chunks, one block per (row pair, kv head, chunk); each writes its partial O (normalised by
// its own sum) and LSE in fp32, the last chunk also runs the tail tiles, and split_merge_kernel
// combines the chunks by LSE -- the same merge that joins the prefix and tail parts.  The whole
// units and the chunks run in one launch (whole units first, so a chunk starts on the first SM
// that frees up).  The forms are separate instantiations (kMode: whole units only, whole units
// then chunks, chunks only), so the common unsplit kernel carries none of the chunk code and a
// launch of chunks only carries none of the whole-unit epilogue.
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace blink {
namespace {

constexpr int BM = 128;       // rows per M tile
constexpr int BN = 128;       // keys per KV tile
constexpr int kSlots = 4;     // K/V ring slots
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kHalfBytes = 128 * 128;  // 128 rows x 128 bytes: one 64-column swizzle panel
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr uint32_t kTmemCols = 512;

constexpr int kMaxRequests = 64;  // blink.py `Batcher.MAX_REQUESTS`

template <int N>
struct IntTag {
    static constexpr int value = N;
};

struct AttnArgs {
    const int32_t *cu;         // [B+1]
    const int32_t *seq_start;  // [B] or nullptr (varlen)
    uint16_t *out;             // [rows, Hq, D]
    float *lse;                // [Hq, rows] or nullptr
    int *err;
    int rows, B, Hq, Hkv, g, tpt, max_tail;
    float scale_log2;
    // Requests: request r owns tail rows [req_row[r], req_row[r+1]) and the prefix of req_P[r]
    // tokens at arena slots [req_pre[r], req_pre[r] + req_P[r]).  Blocks [req_blk[r], req_blk[r+1])
    // work on request r (a block never straddles two requests).
    // Split of the prefix (one request only): with n_split > 1 the prefix tiles of units
    // [unit0, ...) are cut into chunks of split_tiles (the last chunk: the remaining 0 ..
    // split_tiles tiles, plus the tail tiles); unit (row pair, kv head, chunk) writes its
    // partial O (normalised by its own sum) and LSE, the last chunk also runs the tail tiles, and
    // split_merge_kernel then merges the chunks of every row by LSE.
    int n_split, split_tiles;
    // Work units are (row pair, kv head), numbered kv-head-major: u = head * n_pairs + row pair.
    // Block b < unit0 runs unit b whole; block unit0 + j * n_split + c runs chunk c of unit
    // unit0 + j (the chunked instantiation only; the unsplit one runs unit b for every block b).
    int n_pairs, unit0;
    float *part_o;    // [split units][n_split][D / 4][2 BM] float4, split unit = u - unit0 (a column
                      // group's rows contiguous, so a warp's partial stores are coalesced)
    float *part_lse;  // [split units][n_split][2 BM]
    int n_req;
    int req_row[kMaxRequests + 1];
    int req_blk[kMaxRequests + 1];
    int req_pre[kMaxRequests];
    int req_P[kMaxRequests];
};

template <int D>
struct Layout {
    static constexpr int kQTileBytes = BM * D * 2;
    static constexpr int kKVTileBytes = BN * D * 2;
    static constexpr int kPanels = D / 64;
    static constexpr int kQOff0 = 0;
    static constexpr int kQOff1 = kQTileBytes;
    static constexpr int kKVOff = 2 * kQTileBytes;
    static constexpr int kBarOff = kKVOff + kSlots * kKVTileBytes;
    static constexpr int kBytes = kBarOff + 256;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 bytes
};

__device__ __forceinline__ int start_of(const AttnArgs &a, int b)
{
    return a.seq_start ? __ldg(a.seq_start + b) : __ldg(a.cu + b) - __ldg(a.cu);
}
__device__ __forceinline__ int len_of(const AttnArgs &a, int b) { return __ldg(a.cu + b + 1) - __ldg(a.cu + b); }

// Largest b with start_b <= t, or -1.
__device__ __forceinline__ int owner_floor(const AttnArgs &a, int t)
{
    int lo = 0, hi = a.B - 1, ans = -1;
    while (lo <= hi) {
        int mid = (lo + hi) >> 1;
        if (start_of(a, mid) <= t) {
            ans = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    return ans;
}

// The same search by a whole warp (every lane gets the answer): 32 probes per round, so 2-3
// dependent rounds of loads instead of one per halving.  Starts ascend with b.
__device__ __forceinline__ int owner_floor_warp(const AttnArgs &a, int t, int lane)
{
    int lo = 0, n = a.B;  // candidates [lo, lo + n); start_lo <= t once past the first round
    while (n > 32) {
        const int step = (n + 31) / 32;
        const int idx = lo + lane * step;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, idx < lo + n && start_of(a, idx) <= t);
        if (m == 0) return -1;  // the first start is past t
        const int nlo = lo + (31 - __clz(m)) * step;
        n = min(step, lo + n - nlo);
        lo = nlo;
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, lane < n && start_of(a, lo + lane) <= t);
    return m ? lo + 31 - __clz(m) : -1;
}

// Largest b >= b0 with start_b <= t, walking forward from b0 (start_b0 <= t, or b0 = -1); after
// eight steps (many short questions inside one block) it falls back to the binary search.
__device__ __forceinline__ int owner_from(const AttnArgs &a, int t, int b0)
{
    int b = b0;
    for (int steps = 0; b + 1 < a.B && start_of(a, b + 1) <= t; ++b)
        if (++steps > 8) return owner_floor(a, t);
    return b;
}

__device__ __forceinline__ bool question_ok(const AttnArgs &a, int s, int L)
{
    return L >= 1 && L <= a.max_tail && s >= 0 && static_cast<long long>(s) + L <= a.rows;
}

// Masks for the tail tiles.  Keys [J0, J0 + 32) of a row are set to -inf where key < lo or
// key > hi (the row's question start and its own token, relative to the tile).  A 32-key chunk
// that every row of the warp keeps whole is left alone and one that every row drops is cleared,
// so only the chunk a boundary crosses is masked key by key: on a causal diagonal tile that is one
// chunk in four.  The per-key step is written out in PTX (a compare, a compare-or, a predicated
// move of -inf per key) so that the row's 128 scores stay in registers across the branches (the
// same branches in C++ cost 2.4 KB of spills).
#define BLINK_MASK1(k) \
    "setp.gt.s32 p, %32, " #k "; setp.lt.or.s32 p, %33, " #k ", p; @p mov.f32 %" #k ", 0fFF800000;\n\t"
#define BLINK_DROP1(k) "mov.f32 %" #k ", 0fFF800000;\n\t"
#define BLINK_X8(M, a, b, c, d, e, f, g, h) M(a) M(b) M(c) M(d) M(e) M(f) M(g) M(h)
#define BLINK_X32(M)                                                                                           \
    BLINK_X8(M, 0, 1, 2, 3, 4, 5, 6, 7)                                                                        \
    BLINK_X8(M, 8, 9, 10, 11, 12, 13, 14, 15)                                                                  \
    BLINK_X8(M, 16, 17, 18, 19, 20, 21, 22, 23) BLINK_X8(M, 24, 25, 26, 27, 28, 29, 30, 31)
#define BLINK_OPS32(J)                                                                                          \
    "+f"(s[J + 0]), "+f"(s[J + 1]), "+f"(s[J + 2]), "+f"(s[J + 3]), "+f"(s[J + 4]), "+f"(s[J + 5]),             \
        "+f"(s[J + 6]), "+f"(s[J + 7]), "+f"(s[J + 8]), "+f"(s[J + 9]), "+f"(s[J + 10]), "+f"(s[J + 11]),       \
        "+f"(s[J + 12]), "+f"(s[J + 13]), "+f"(s[J + 14]), "+f"(s[J + 15]), "+f"(s[J + 16]), "+f"(s[J + 17]),   \
        "+f"(s[J + 18]), "+f"(s[J + 19]), "+f"(s[J + 20]), "+f"(s[J + 21]), "+f"(s[J + 22]), "+f"(s[J + 23]),   \
        "+f"(s[J + 24]), "+f"(s[J + 25]), "+f"(s[J + 26]), "+f"(s[J + 27]), "+f"(s[J + 28]), "+f"(s[J + 29]),   \
        "+f"(s[J + 30]), "+f"(s[J + 31])

template <int J0>
__device__ __forceinline__ void mask_chunk(float (&s)[BN], int lo, int hi)
{
    if (__all_sync(0xFFFFFFFFu, lo <= J0 && hi >= J0 + 31)) return;
    if (__all_sync(0xFFFFFFFFu, hi < J0 || lo > J0 + 31)) {
        asm volatile("{\n\t" BLINK_X32(BLINK_DROP1) "}" : BLINK_OPS32(J0));
    } else {
        const int dlo = lo - J0, dhi = hi - J0;  // key k of the chunk is dropped if k < dlo or k > dhi
        asm volatile("{\n\t.reg .pred p;\n\t" BLINK_X32(BLINK_MASK1) "}" : BLINK_OPS32(J0) : "r"(dlo), "r"(dhi));
    }
}

// Every tail-tile mask of a row: its keys below lo or above hi.
__device__ __forceinline__ void mask_tail_tile(float (&s)[BN], int lo, int hi)
{
    if (__all_sync(0xFFFFFFFFu, lo <= 0 && hi >= BN - 1)) return;  // most tiles of a long causal tail
    mask_chunk<0>(s, lo, hi);
    mask_chunk<32>(s, lo, hi);
    mask_chunk<64>(s, lo, hi);
    mask_chunk<96>(s, lo, hi);
}
#undef BLINK_MASK1
#undef BLINK_DROP1
#undef BLINK_X8
#undef BLINK_X32
#undef BLINK_OPS32

// kMode 0: whole units only (the chunk arithmetic folds away: the plain kernel); 1: whole units,
// then prefix chunks (n_split > 1) that write partial results; 2: prefix chunks only.
constexpr int kWholeUnits = 0, kUnitsThenChunks = 1, kChunksOnly = 2;
template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kpre,
                     const __grid_constant__ CUtensorMap tm_vpre, const __grid_constant__ CUtensorMap tm_ktail,
                     const __grid_constant__ CUtensorMap tm_vtail, const AttnArgs a)
{
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s0 = base + L::kQOff0;
    uint8_t *q_s1 = base + L::kQOff1;
    uint8_t *kv_s = base + L::kKVOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + L::kBarOff);
    uint64_t *q_full = bars + 0;
    uint64_t *full = bars + 1;     // [2] by iteration parity: that iteration's K and V tiles
    uint64_t *empty = bars + 5;    // [4] per ring slot
    uint64_t *s_full = bars + 9;   // [2]
    uint64_t *p_full = bars + 11;  // [2]
    uint64_t *o_full = bars + 13;  // [2]
    uint64_t *mma_done = bars + 15;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 16);
    int *sched = reinterpret_cast<int *>(tmem_holder + 1);  // kbeg, n_tail, abort, first owner
    volatile int *abort_flag = sched + 2;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bid = static_cast<int>(blockIdx.x);
    constexpr bool kSplit = kMode != kWholeUnits;
    const bool chunk = kMode == kChunksOnly || (kMode == kUnitsThenChunks && bid >= a.unit0);  // not a whole unit
    const int local = chunk ? (bid - a.unit0) / a.n_split : 0;       // split unit
    const int split = chunk ? (bid - a.unit0) % a.n_split : 0;       // prefix chunk
    const int unit = chunk ? a.unit0 + local : bid;
    const int head = unit / a.n_pairs;
    const int bx = unit - head * a.n_pairs;  // row pair
    int req = 0;  // this block's request
    while (req + 1 < a.n_req && a.req_blk[req + 1] <= bx) ++req;
    const int req_begin = a.req_row[req], req_end = a.req_row[req + 1];
    const int P = a.req_P[req], pre_start = a.req_pre[req];
    const int pre_lo = chunk ? split * a.split_tiles : 0;  // first prefix tile of this unit
    const int n_pre = chunk ? max(0, min((P + BN - 1) / BN - pre_lo, a.split_tiles)) : (P + BN - 1) / BN;
    const bool has_tail = !chunk || split == a.n_split - 1;
    const int n_early = min(n_pre, kSlots / 2);  // prefix iterations copied before the tail search
    // Within a request the blocks run from the last row pair to the first: with a causal tail the
    // late pairs have the most keys, and starting them first shortens the end of the launch.
    const int t0 = req_begin + (a.req_blk[req + 1] - 1 - bx) * 2 * a.tpt;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            ptx::mbar_init(q_full, 1);
            for (int i = 0; i < 2; ++i) ptx::mbar_init(full + i, 2);  // the K and the V copy
            for (int i = 0; i < kSlots; ++i) ptx::mbar_init(empty + i, 1);
            for (int t = 0; t < 2; ++t) {
                ptx::mbar_init(s_full + t, 1);
                ptx::mbar_init(p_full + t, 128);
                ptx::mbar_init(o_full + t, 1);
            }
            ptx::mbar_init(mma_done, 1);
            ptx::fence_mbar_init();
            sched[2] = 0;
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_kpre);
            ptx::tma_prefetch_desc(&tm_vpre);
            ptx::tma_prefetch_desc(&tm_ktail);
            ptx::tma_prefetch_desc(&tm_vtail);
            // The Q tiles need no schedule: request them first.  The second tile is loaded only
            // if it starts inside the request (its rows past the tensor's end are then
            // zero-filled by the copy); otherwise its rows stay as they are and are never stored.
            // (Rows past g * tpt, zeroed below by the other warps, are outside the copied box.)
            const uint32_t q_box = 64u * a.g * a.tpt * 2u;
            const int q_tiles = (t0 + a.tpt < req_end) ? 2 : 1;
            ptx::mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(q_tiles) * L::kPanels * q_box);
            for (int t = 0; t < q_tiles; ++t)
                for (int p = 0; p < L::kPanels; ++p)
                    ptx::tma_load_3d((t == 0 ? q_s0 : q_s1) + p * kHalfBytes, &tm_q, p * 64, head * a.g,
                                     t0 + t * a.tpt, q_full);
            // The first prefix tiles need no schedule either: their copies run during the search
            // for the block's tail keys below (the ring's first slots are free).
            for (int it = 0; it < n_early; ++it) {
                uint64_t *stage_full = full + (it & 1);
                const int kb = pre_start + (pre_lo + it) * BN;
                for (int kv = 0; kv < 2; ++kv) {
                    ptx::mbar_arrive_expect_tx(stage_full, L::kKVTileBytes);
                    for (int p = 0; p < L::kPanels; ++p)
                        ptx::tma_load_3d(kv_s + (2 * it + kv) * L::kKVTileBytes + p * kHalfBytes,
                                         kv ? &tm_vpre : &tm_kpre, p * 64, head, kb, stage_full);
                }
            }
        }
        __syncwarp();
        // Tail keys this block needs: from the start of the first question it touches.
        const int t_end = min(t0 + 2 * a.tpt, req_end);
        int kbeg = -1;
        const int b = owner_floor_warp(a, t0, lane);
        if (b >= 0) {
            const int s = start_of(a, b), len = len_of(a, b);
            if (!question_ok(a, s, len) || (t0 < s + len && s < req_begin)) {
                if (lane == 0) atomicCAS(a.err, 0, BLINK_DEVICE_FLAG);
            } else if (t0 < s + len) {
                kbeg = s;
            }
        }
        if (kbeg < 0 && b + 1 < a.B) {
            const int s = start_of(a, b + 1);
            if (s >= 0 && s < t_end) kbeg = s;
        }
        int n_tail = 0;
        if (kbeg >= 0 && kbeg < t_end) n_tail = (t_end - kbeg + BN - 1) / BN;
        if (lane == 0) {
            sched[0] = kbeg < 0 ? 0 : kbeg;
            sched[1] = has_tail ? n_tail : 0;
            sched[3] = b;  // owner of the block's first token, where the softmax rows' searches start
        }
    }
    if (warp == 0) {
        ptx::tmem_alloc(tmem_holder, kTmemCols);
        ptx::tmem_relinquish();
    }
    // Rows of a Q tile past g * tpt are never loaded: zero them so they stay finite.
    const int rows_used = a.g * a.tpt;
    if (warp < 8 && rows_used < BM) {
        const int pad_bytes = (BM - rows_used) * 128;
        for (int t = 0; t < 2; ++t) {
            uint8_t *q = t == 0 ? q_s0 : q_s1;
            for (int p = 0; p < L::kPanels; ++p) {
                uint8_t *dst = q + p * kHalfBytes + rows_used * 128;
                for (int off = threadIdx.x * 16; off < pad_bytes; off += 256 * 16)
                    *reinterpret_cast<uint4 *>(dst + off) = make_uint4(0, 0, 0, 0);
            }
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    const uint32_t tmem = *tmem_holder;
    const int kbeg = sched[0];
    const int n_iter = n_pre + sched[1];

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- TMA producer
        // K and V of iteration it go to slots 2 (it & 1) and 2 (it & 1) + 1 and both complete on
        // full[it & 1], so the MMA thread waits once per iteration for its operands; each slot is
        // released on its own (K after S_1, V after the product P_1 V) so neither copy waits for
        // the other's use.
        if (lane == 0) {
            int n = 2 * n_early;
            for (int it = n_early; it < n_iter; ++it) {
                const bool pre = it < n_pre;
                const int kb = pre ? pre_start + (pre_lo + it) * BN : kbeg + (it - n_pre) * BN;
                uint64_t *stage_full = full + (it & 1);
                bool ok = true;
                for (int kv = 0; kv < 2; ++kv) {
                    const int slot = n % kSlots;
                    const uint32_t ph = (n / kSlots) & 1;
                    if (!ptx::mbar_wait(empty + slot, ph ^ 1u, abort_flag, a.err, BLINK_DEVICE_TIMEOUT)) {
                        // giving up after the K copy: complete the iteration's arrival count so that
                        // the drain below still sees that copy land
                        if (kv == 1) ptx::mbar_arrive(stage_full);
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(stage_full, L::kKVTileBytes);
                    const CUtensorMap *map = pre ? (kv ? &tm_vpre : &tm_kpre) : (kv ? &tm_vtail : &tm_ktail);
                    for (int p = 0; p < L::kPanels; ++p)
                        ptx::tma_load_3d(kv_s + slot * L::kKVTileBytes + p * kHalfBytes, map, p * 64, head, kb,
                                         stage_full);
                    ++n;
                }
                if (!ok) break;
            }
            // The merge of the chunks is this launch's programmatic dependent: let it be scheduled
            // once every block is this close to its end (it waits for the grid's end to read).
            if constexpr (kSplit) ptx::grid_launch_dependents();
            // Drain: every copy issued must have landed before the block may exit.  Copies of
            // iterations before the last two were waited for by the MMA thread before their slots
            // were reused.
            volatile int no_abort = 0;
            ptx::mbar_wait(q_full, 0, &no_abort, a.err, BLINK_DEVICE_TIMEOUT);
            const int n_it = (n + 1) / 2;  // iterations with at least their K copy issued
            for (int j = n_it > 2 ? n_it - 2 : 0; j < n_it; ++j) {
                no_abort = 0;
                ptx::mbar_wait(full + (j & 1), (j >> 1) & 1, &no_abort, a.err, BLINK_DEVICE_TIMEOUT);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        // The tensor core takes a product about when the previous one finishes, so whatever this
        // thread does between two issues is idle tensor time: every operand address is built
        // before the loop, the loop is unrolled by two so that the ring slots (K in 0 or 2, V in
        // 1 or 3, by the iteration's parity) are compile-time, and each group of 8 products is
        // issued from one asm block.
        if (lane == 0) {
            constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(BM, D, true);
            const uint32_t s_col[2] = {0u, 128u};
            const uint32_t o_col[2] = {256u, 256u + D};
            const uint32_t q_addr[2] = {ptx::smem_u32(q_s0), ptx::smem_u32(q_s1)};
            const uint32_t kv_addr = ptx::smem_u32(kv_s);
            uint64_t qd[2][D / 16], kd[2][D / 16], vd[2][BN / 16];
            uint32_t pa[2][BN / 16];  // P_t columns of each k-step (bf16 pairs: 8 columns per 16 keys)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                qd[0][kk] = ptx::smem_desc_sw128(q_addr[0] + off, 16, 1024);
                qd[1][kk] = ptx::smem_desc_sw128(q_addr[1] + off, 16, 1024);
                kd[0][kk] = ptx::smem_desc_sw128(kv_addr + 0 * L::kKVTileBytes + off, 16, 1024);
                kd[1][kk] = ptx::smem_desc_sw128(kv_addr + 2 * L::kKVTileBytes + off, 16, 1024);
            }
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
                vd[0][kk] = ptx::smem_desc_sw128(kv_addr + 1 * L::kKVTileBytes + kk * 2048, kHalfBytes, 1024);
                vd[1][kk] = ptx::smem_desc_sw128(kv_addr + 3 * L::kKVTileBytes + kk * 2048, kHalfBytes, 1024);
                pa[0][kk] = tmem + s_col[0] + kk * 8;
                pa[1][kk] = tmem + s_col[1] + kk * 8;
            }
            auto qk = [&](int t, int par) {
                if constexpr (D == 128) {
                    ptx::mma_ss_x8(tmem + s_col[t], qd[t], kd[par], idesc_s, 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        ptx::mma_ss(tmem + s_col[t], qd[t][kk], kd[par][kk], idesc_s, kk > 0 ? 1u : 0u);
                }
            };
            auto pv = [&](int t, int par, bool first) {
                ptx::mma_ts_x8(tmem + o_col[t], pa[t], vd[par], idesc_pv, first ? 0u : 1u);
            };
            // One KV iteration; kPar = i & 1 selects the slots.
            auto step = [&](auto par_tag, int i) -> bool {
                constexpr int kPar = decltype(par_tag)::value;
                constexpr int kslot = 2 * kPar, prev_vslot = 3 - 2 * kPar;
                // K and V of this iteration (one barrier per iteration parity)
                if (!ptx::mbar_wait(full + kPar, (i >> 1) & 1, abort_flag, a.err, BLINK_DEVICE_TIMEOUT)) return false;
                ptx::tc_fence_after();
                qk(0, kPar);
                ptx::mma_commit(s_full + 0);
                if (i > 0) {
                    if (!ptx::mbar_wait(p_full + 1, (i - 1) & 1, abort_flag, a.err, BLINK_DEVICE_TIMEOUT))
                        return false;
                    ptx::tc_fence_after();
                    pv(1, 1 - kPar, i == 1);
                    ptx::mma_commit(empty + prev_vslot);
                }
                qk(1, kPar);
                ptx::mma_commit(s_full + 1);
                ptx::mma_commit(empty + kslot);
                if (!ptx::mbar_wait(p_full + 0, i & 1, abort_flag, a.err, BLINK_DEVICE_TIMEOUT)) return false;
                ptx::tc_fence_after();
                pv(0, kPar, i == 0);
                if (i == n_iter - 1) ptx::mma_commit(o_full + 0);
                return true;
            };
            bool ok = ptx::mbar_wait(q_full, 0, abort_flag, a.err, BLINK_DEVICE_TIMEOUT);
            ptx::tc_fence_after();
            for (int i = 0; ok && i < n_iter; i += 2) {
                ok = step(IntTag<0>{}, i);
                if (ok && i + 1 < n_iter) ok = step(IntTag<1>{}, i + 1);
            }
            if (ok) {
                if (n_iter > 0) {
                    const int i = n_iter - 1;
                    const int vslot = (2 * i + 1) % kSlots;
                    if (ptx::mbar_wait(p_full + 1, i & 1, abort_flag, a.err, BLINK_DEVICE_TIMEOUT)) {
                        ptx::tc_fence_after();
                        if (i & 1)
                            pv(1, 1, i == 0);
                        else
                            pv(1, 0, i == 0);
                        ptx::mma_commit(empty + vslot);
                        ptx::mma_commit(o_full + 1);
                    }
                } else {
                    ptx::mma_commit(o_full + 0);
                    ptx::mma_commit(o_full + 1);
                }
            }
            // Every MMA issued must be complete before tensor memory is released.
            ptx::mma_commit(mma_done);
            volatile int no_abort = 0;
            ptx::mbar_wait(mma_done, 0, &no_abort, a.err, BLINK_DEVICE_TIMEOUT);
        }
    } else {
        // ---------------------------------------------------------------- softmax (one row per thread)
        const int t = warp >> 2;              // which of the two M tiles
        const int r = (warp & 3) * 32 + lane;  // row inside the tile = TMEM lane
        const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_col = t * 128u;
        const uint32_t o_col = 256u + t * D;
        const int tok = t0 + t * a.tpt + r / a.g;
        const int hq = head * a.g + r % a.g;
        const bool row_ok = r < rows_used && tok < req_end;
        bool owned = false;
        int q_lo = 0;
        if (row_ok) {
            const int b = owner_from(a, tok, sched[3]);
            if (b >= 0) {
                const int s = start_of(a, b), len = len_of(a, b);
                if (!question_ok(a, s, len) || (tok < s + len && s < req_begin)) {
                    atomicCAS(a.err, 0, BLINK_DEVICE_FLAG);
                } else if (tok < s + len) {
                    owned = true;
                    q_lo = s;
                }
            }
        }
        const float sl2 = a.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < n_iter; ++i) {
            if (!(ok = ptx::mbar_wait(s_full + t, i & 1, abort_flag, a.err, BLINK_DEVICE_TIMEOUT))) break;
            ptx::tc_fence_after();
            float s[BN];
            {
                uint32_t raw[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
                    ptx::tmem_ld32(trow + s_col + c * 32, *reinterpret_cast<uint32_t(*)[32]>(raw + c * 32));
                ptx::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < BN; ++j) s[j] = __uint_as_float(raw[j]);
            }
            // masks
            if (i < n_pre) {
                const int kb = (pre_lo + i) * BN;
                if (kb + BN > P) {
                    const int lim = P - kb;
#pragma unroll
                    for (int j = 0; j < BN; ++j)
                        if (j >= lim) s[j] = -INFINITY;
                }
            } else {
                const int kb = kbeg + (i - n_pre) * BN;
                const int lo_j = q_lo - kb;
                const int hi_j = owned ? tok - kb : -1;
                mask_tail_tile(s, lo_j, hi_j);
            }
            // row max, three operands per instruction, four independent chains
            float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]), mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
            for (int j = 8; j < BN; j += 8) {
                mx0 = ptx::max3(mx0, s[j], s[j + 1]);
                mx1 = ptx::max3(mx1, s[j + 2], s[j + 3]);
                mx2 = ptx::max3(mx2, s[j + 4], s[j + 5]);
                mx3 = ptx::max3(mx3, s[j + 6], s[j + 7]);
            }
            const float m_new = fmaxf(m, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2);
            const bool need = m_new > m + kRescaleThreshold;
            const bool rescale = __any_sync(0xFFFFFFFFu, need);  // warp-uniform: TMEM access is collective
            float alpha = 1.f;
            if (rescale) {
                alpha = (m == -INFINITY) ? 0.f : ptx::ex2(m - m_new);
                l *= alpha;
                m = m_new;
            }
            const float m_use = (m == -INFINITY) ? 0.f : m;
            if constexpr (D == 128) {
                // The softmax warps are bound by instruction issue, not by the exp2 unit: the
                // exponent arguments of an element pair take one f32x2 fma (bit-identical to two
                // fmaf), and four row-sum chains keep the adds from waiting on each other.
                const uint64_t sl2x2 = ptx::f32x2(sl2, sl2), negm_x2 = ptx::f32x2(-m_use, -m_use);
                float rs0 = 0.f, rs1 = 0.f, rs2 = 0.f, rs3 = 0.f;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pk[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const uint64_t s2 = ptx::f32x2(s[c * 64 + 2 * j], s[c * 64 + 2 * j + 1]);
                        float x0, x1;
                        ptx::f32x2_split(ptx::fma_f32x2(s2, sl2x2, negm_x2), x0, x1);
                        const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                        if (j & 1) {
                            rs2 += p0;
                            rs3 += p1;
                        } else {
                            rs0 += p0;
                            rs1 += p1;
                        }
                        pk[j] = ptx::pack_bf16x2(p0, p1);
                    }
                    ptx::tmem_st32(trow + s_col + c * 32, pk);
                }
                l += (rs0 + rs2) + (rs1 + rs3);
            } else {  // d = 64: the scalar form (the packed one costs this instantiation spills)
                float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pk[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float p0 = ptx::ex2(fmaf(s[c * 64 + 2 * j], sl2, -m_use));
                        const float p1 = ptx::ex2(fmaf(s[c * 64 + 2 * j + 1], sl2, -m_use));
                        rs0 += p0;
                        rs1 += p1;
                        pk[j] = ptx::pack_bf16x2(p0, p1);
                    }
                    ptx::tmem_st32(trow + s_col + c * 32, pk);
                }
                l += rs0 + rs1;
            }
            // O_t still holds the sum up to the previous tile (that product completed before this
            // tile's scores were signalled); scale it to the new max before P_t is released.
            if (rescale && i > 0) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld32(trow + o_col + c * 32, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    ptx::tmem_st32(trow + o_col + c * 32, o);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(p_full + t);
        }
        // epilogue: O / l -> bf16 (or, for a prefix chunk, the partial O / l in fp32 and its LSE)
        if (ok && ptx::mbar_wait(o_full + t, 0, abort_flag, a.err, BLINK_DEVICE_TIMEOUT)) {
            ptx::tc_fence_after();
            const float inv = (owned && l > 0.f) ? 1.0f / l : 0.f;
            const float row_lse =
                (owned && l > 0.f) ? (((m == -INFINITY) ? 0.f : m) + __log2f(l)) * kLn2 : -INFINITY;
            const bool partial = chunk;
            const int64_t prow = (static_cast<int64_t>(local) * a.n_split + split) * (2 * BM) + t * BM + r;
            uint16_t *dst = a.out + (static_cast<int64_t>(tok) * a.Hq + hq) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (n_iter > 0) {
                    ptx::tmem_ld32(trow + o_col + c * 32, o);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0u;
                }
                if (row_ok && partial) {
                    // float4 group g of this row at [unit, chunk, g, row]
                    float4 *p4 = reinterpret_cast<float4 *>(a.part_o) +
                                 ((prow - (t * BM + r)) / (2 * BM) * (D / 4) + c * 8) * (2 * BM) + t * BM + r;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        p4[j * (2 * BM)] = make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                                                       __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
                } else if (row_ok) {
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        pk[j] = ptx::pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
                    for (int j = 0; j < 4; ++j) d4[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                }
            }
            if (row_ok && partial) {
                a.part_lse[prow] = row_lse;
            } else if (row_ok && a.lse) {
                a.lse[static_cast<int64_t>(hq) * a.rows + tok] = row_lse;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// Single-tile form for very short work: one 128-row M tile per block, a 2-slot K/V ring and 256
// tensor-memory columns (S, O), so two blocks share an SM.  Their serial S -> softmax -> P V
// chains interleave on the tensor core (the job the two-tile ping-pong does inside one block),
// and one block's start and epilogue overlap the other's work.  Same masks, merge and request
// table as the two-tile kernel.
// ---------------------------------------------------------------------------------------------
constexpr int kThreads1 = 192;  // 4 softmax warps, the TMA producer, the MMA issuer
constexpr int kProducerWarp1 = 4;
constexpr int kMmaWarp1 = 5;
constexpr uint32_t kTmemCols1 = 256;

template <int D>
struct Layout1 {
    static constexpr int kQTileBytes = BM * D * 2;
    static constexpr int kKVTileBytes = BN * D * 2;
    static constexpr int kPanels = D / 64;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = kQTileBytes;  // slot 0: K, slot 1: V
    static constexpr int kBarOff = kKVOff + 2 * kKVTileBytes;
    static constexpr int kBytes = kBarOff + 256;
    static constexpr int kAlloc = kBytes + 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads1, 2)
    attention_single_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kpre,
                            const __grid_constant__ CUtensorMap tm_vpre, const __grid_constant__ CUtensorMap tm_ktail,
                            const __grid_constant__ CUtensorMap tm_vtail, const AttnArgs a)
{
    using L = Layout1<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = base + L::kQOff;
    uint8_t *kv_s = base + L::kKVOff;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + L::kBarOff);
    uint64_t *q_full = bars + 0;
    uint64_t *full = bars + 1;   // [2]
    uint64_t *empty = bars + 3;  // [2]
    uint64_t *s_full = bars + 5;
    uint64_t *p_full = bars + 6;
    uint64_t *o_full = bars + 7;
    uint64_t *mma_done = bars + 8;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 9);
    int *sched = reinterpret_cast<int *>(tmem_holder + 1);  // kbeg, n_tail, abort, first owner
    volatile int *abort_flag = sched + 2;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int head = blockIdx.y;
    const int bx = static_cast<int>(blockIdx.x);
    int req = 0;
    while (req + 1 < a.n_req && a.req_blk[req + 1] <= bx) ++req;
    const int req_begin = a.req_row[req], req_end = a.req_row[req + 1];
    const int P = a.req_P[req], pre_start = a.req_pre[req];
    const int n_pre = (P + BN - 1) / BN;
    // last tile of the request first: with a causal tail the late tiles have the most keys
    const int t0 = req_begin + (a.req_blk[req + 1] - 1 - bx) * a.tpt;

    if (warp == kProducerWarp1) {
        if (lane == 0) {
            ptx::mbar_init(q_full, 1);
            for (int i = 0; i < 2; ++i) {
                ptx::mbar_init(full + i, 1);
                ptx::mbar_init(empty + i, 1);
            }
            ptx::mbar_init(s_full, 1);
            ptx::mbar_init(p_full, 128);
            ptx::mbar_init(o_full, 1);
            ptx::mbar_init(mma_done, 1);
            ptx::fence_mbar_init();
            sched[2] = 0;
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_kpre);
            ptx::tma_prefetch_desc(&tm_vpre);
            ptx::tma_prefetch_desc(&tm_ktail);
            ptx::tma_prefetch_desc(&tm_vtail);
            // Q first: it needs no schedule (rows past the tensor's end are zero-filled)
            const uint32_t q_box = 64u * a.g * a.tpt * 2u;
            ptx::mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(L::kPanels) * q_box);
            for (int p = 0; p < L::kPanels; ++p)
                ptx::tma_load_3d(q_s + p * kHalfBytes, &tm_q, p * 64, head * a.g, t0, q_full);
        }
        __syncwarp();
        const int t_end = min(t0 + a.tpt, req_end);
        int kbeg = -1;
        const int b = owner_floor_warp(a, t0, lane);
        if (b >= 0) {
            const int s = start_of(a, b), len = len_of(a, b);
            if (!question_ok(a, s, len) || (t0 < s + len && s < req_begin)) {
                if (lane == 0) atomicCAS(a.err, 0, BLINK_DEVICE_FLAG);
            } else if (t0 < s + len) {
                kbeg = s;
            }
        }
        if (kbeg < 0 && b + 1 < a.B) {
            const int s = start_of(a, b + 1);
            if (s >= 0 && s < t_end) kbeg = s;
        }
        int n_tail = 0;
        if (kbeg >= 0 && kbeg < t_end) n_tail = (t_end - kbeg + BN - 1) / BN;
        if (lane == 0) {
            sched[0] = kbeg < 0 ? 0 : kbeg;
            sched[1] = n_tail;
            sched[3] = b;
        }
    }
    if (warp == 0) {
        ptx::tmem_alloc(tmem_holder, kTmemCols1);
        ptx::tmem_relinquish();
    }
    const int rows_used = a.g * a.tpt;
    if (warp < 4 && rows_used < BM) {  // rows of the Q tile past g * tpt are never loaded
        const int pad_bytes = (BM - rows_used) * 128;
        for (int p = 0; p < L::kPanels; ++p) {
            uint8_t *dst = q_s + p * kHalfBytes + rows_used * 128;
            for (int off = threadIdx.x * 16; off < pad_bytes; off += 128 * 16)
                *reinterpret_cast<uint4 *>(dst + off) = make_uint4(0, 0, 0, 0);
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    const uint32_t tmem = *tmem_holder;
    const int kbeg = sched[0];
    const int n_iter = n_pre + sched[1];

    if (warp == kProducerWarp1) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            bool ok = true;
            int issued[2] = {0, 0};  // K and V tiles issued
            for (int it = 0; ok && it < n_iter; ++it) {
                const bool pre = it < n_pre;
                const int kb = pre ? pre_start + it * BN : kbeg + (it - n_pre) * BN;
                for (int kv = 0; kv < 2; ++kv) {  // K into slot 0, V into slot 1
                    if (!(ok = ptx::mbar_wait(empty + kv, (it & 1) ^ 1u, abort_flag, a.err, BLINK_DEVICE_TIMEOUT)))
                        break;
                    ++issued[kv];
                    ptx::mbar_arrive_expect_tx(full + kv, L::kKVTileBytes);
                    const CUtensorMap *map = pre ? (kv ? &tm_vpre : &tm_kpre) : (kv ? &tm_vtail : &tm_ktail);
                    for (int p = 0; p < L::kPanels; ++p)
                        ptx::tma_load_3d(kv_s + kv * L::kKVTileBytes + p * kHalfBytes, map, p * 64, head, kb,
                                         full + kv);
                }
            }
            // Drain: every copy issued must have landed before the block may exit.
            volatile int no_abort = 0;
            ptx::mbar_wait(q_full, 0, &no_abort, a.err, BLINK_DEVICE_TIMEOUT);
            for (int kv = 0; kv < 2; ++kv) {  // the last tile issued to each slot
                if (issued[kv] == 0) continue;
                no_abort = 0;
                ptx::mbar_wait(full + kv, (issued[kv] - 1) & 1, &no_abort, a.err, BLINK_DEVICE_TIMEOUT);
            }
        }
    } else if (warp == kMmaWarp1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(BM, D, true);
            const uint32_t q_addr = ptx::smem_u32(q_s), k_addr = ptx::smem_u32(kv_s);
            const uint32_t v_addr = k_addr + L::kKVTileBytes;
            uint64_t qd[D / 16], kd[D / 16], vd[BN / 16];
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                qd[kk] = ptx::smem_desc_sw128(q_addr + off, 16, 1024);
                kd[kk] = ptx::smem_desc_sw128(k_addr + off, 16, 1024);
            }
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) vd[kk] = ptx::smem_desc_sw128(v_addr + kk * 2048, kHalfBytes, 1024);
            const uint32_t s_col = 0u, o_col = 128u;
            bool ok = ptx::mbar_wait(q_full, 0, abort_flag, a.err, BLINK_DEVICE_TIMEOUT);
            ptx::tc_fence_after();
            for (int i = 0; ok && i < n_iter; ++i) {
                if (!(ok = ptx::mbar_wait(full + 0, i & 1, abort_flag, a.err, BLINK_DEVICE_TIMEOUT))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + s_col, qd[kk], kd[kk], idesc_s, kk > 0 ? 1u : 0u);
                ptx::mma_commit(s_full);
                ptx::mma_commit(empty + 0);
                if (!(ok = ptx::mbar_wait(p_full, i & 1, abort_flag, a.err, BLINK_DEVICE_TIMEOUT))) break;
                if (!(ok = ptx::mbar_wait(full + 1, i & 1, abort_flag, a.err, BLINK_DEVICE_TIMEOUT))) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    ptx::mma_ts(tmem + o_col, tmem + s_col + kk * 8, vd[kk], idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(empty + 1);
            }
            if (ok) ptx::mma_commit(o_full);
            ptx::mma_commit(mma_done);
            volatile int no_abort = 0;
            ptx::mbar_wait(mma_done, 0, &no_abort, a.err, BLINK_DEVICE_TIMEOUT);
        }
    } else {
        // ---------------------------------------------------------------- softmax (one row per thread)
        const int r = warp * 32 + lane;  // row of the tile = TMEM lane
        const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const uint32_t s_col = 0u, o_col = 128u;
        const int tok = t0 + r / a.g;
        const int hq = head * a.g + r % a.g;
        const bool row_ok = r < rows_used && tok < req_end;
        bool owned = false;
        int q_lo = 0;
        if (row_ok) {
            const int b = owner_from(a, tok, sched[3]);
            if (b >= 0) {
                const int s = start_of(a, b), len = len_of(a, b);
                if (!question_ok(a, s, len) || (tok < s + len && s < req_begin)) {
                    atomicCAS(a.err, 0, BLINK_DEVICE_FLAG);
                } else if (tok < s + len) {
                    owned = true;
                    q_lo = s;
                }
            }
        }
        const float sl2 = a.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < n_iter; ++i) {
            if (!(ok = ptx::mbar_wait(s_full, i & 1, abort_flag, a.err, BLINK_DEVICE_TIMEOUT))) break;
            ptx::tc_fence_after();
            float s[BN];
            {
                uint32_t raw[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
                    ptx::tmem_ld32(trow + s_col + c * 32, *reinterpret_cast<uint32_t(*)[32]>(raw + c * 32));
                ptx::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < BN; ++j) s[j] = __uint_as_float(raw[j]);
            }
            if (i < n_pre) {
                const int kb = i * BN;
                if (kb + BN > P) {
                    const int lim = P - kb;
#pragma unroll
                    for (int j = 0; j < BN; ++j)
                        if (j >= lim) s[j] = -INFINITY;
                }
            } else {
                const int kb = kbeg + (i - n_pre) * BN;
                const int lo_j = q_lo - kb;
                const int hi_j = owned ? tok - kb : -1;
                mask_tail_tile(s, lo_j, hi_j);
            }
            float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
            for (int j = 4; j < BN; j += 4) {
                mx0 = fmaxf(mx0, s[j]);
                mx1 = fmaxf(mx1, s[j + 1]);
                mx2 = fmaxf(mx2, s[j + 2]);
                mx3 = fmaxf(mx3, s[j + 3]);
            }
            const float m_new = fmaxf(m, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2);
            const bool need = m_new > m + kRescaleThreshold;
            const bool rescale = __any_sync(0xFFFFFFFFu, need);
            float alpha = 1.f;
            if (rescale) {
                alpha = (m == -INFINITY) ? 0.f : ptx::ex2(m - m_new);
                l *= alpha;
                m = m_new;
            }
            const float m_use = (m == -INFINITY) ? 0.f : m;
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float p0 = ptx::ex2(fmaf(s[c * 64 + 2 * j], sl2, -m_use));
                    const float p1 = ptx::ex2(fmaf(s[c * 64 + 2 * j + 1], sl2, -m_use));
                    rs0 += p0;
                    rs1 += p1;
                    pk[j] = ptx::pack_bf16x2(p0, p1);
                }
                ptx::tmem_st32(trow + s_col + c * 32, pk);
            }
            l += rs0 + rs1;
            // O holds the sum up to the previous tile (that product completed before this
            // tile's scores were signalled); scale it to the new max before P is released.
            if (rescale && i > 0) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld32(trow + o_col + c * 32, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    ptx::tmem_st32(trow + o_col + c * 32, o);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(p_full);
        }
        if (ok && ptx::mbar_wait(o_full, 0, abort_flag, a.err, BLINK_DEVICE_TIMEOUT)) {
            ptx::tc_fence_after();
            const float inv = (owned && l > 0.f) ? 1.0f / l : 0.f;
            uint16_t *dst = a.out + (static_cast<int64_t>(tok) * a.Hq + hq) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (n_iter > 0) {
                    ptx::tmem_ld32(trow + o_col + c * 32, o);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0u;
                }
                if (row_ok) {
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        pk[j] = ptx::pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
                    // 32-byte stores: a warp's 32 rows land in 32 places, so each store should at
                    // least fill a whole DRAM sector (measured 3 % faster on short causal work; in
                    // the two-tile kernel the extra registers cost spills and 1 %)
                    uint16_t *d8 = dst + c * 32;
                    ptx::st_global_v8(d8, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
                    ptx::st_global_v8(d8 + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
                }
            }
            if (row_ok && a.lse) {
                const float v = (owned && l > 0.f) ? (((m == -INFINITY) ? 0.f : m) + __log2f(l)) * kLn2 : -INFINITY;
                a.lse[static_cast<int64_t>(hq) * a.rows + tok] = v;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols1);
}

// Merge of the prefix chunks (one request).  Thread = (row of a row pair's two M tiles, 8
// output columns); a block covers 16 rows of one unit (u = row pair * Hkv + kv head) and the
// 16 threads of one column group take consecutive rows, reading the partials (stored column
// group by column group) as contiguous runs.  O = sum_c w_c O_c / sum_c w_c with
// w_c = exp(lse_c - max_c lse_c); the LSE (written by each row's first column group) is
// max + log(sum w).  Launched as the attention launch's programmatic dependent, so its blocks may
// be resident before that launch ends; each waits for the attention grid's end (and the
// visibility of its partials) before it reads anything.
constexpr int kMergeRows = 16;  // rows per merge block

template <int D, int kGroup>
__global__ void __launch_bounds__(kMergeRows * (D / 8))
    split_merge_kernel(const AttnArgs a, int nb)
{
    ptx::grid_dep_wait();  // every block, before any read or early return
    const int local = blockIdx.x / (2 * BM / kMergeRows);  // split unit
    const int rr = (blockIdx.x % (2 * BM / kMergeRows)) * kMergeRows + threadIdx.x % kMergeRows;  // row of the pair
    const int cg = threadIdx.x / kMergeRows;
    const int unit = a.unit0 + local;
    const int head = unit / a.n_pairs, bx = unit - head * a.n_pairs;
    const int t = rr / BM, r = rr % BM;
    const int t0 = (nb - 1 - bx) * 2 * a.tpt;
    const int tok = t0 + t * a.tpt + r / a.g;
    const int hq = head * a.g + r % a.g;
    if (r >= a.g * a.tpt || tok >= a.rows) return;
    const int S = a.n_split;
    const int64_t row0 = static_cast<int64_t>(local) * S * (2 * BM) + rr;
    // One pass over the chunks in groups of kGroup: a group's LSE and O loads are all issued
    // before any is used (one L2 round trip per group), and the running sums are rescaled to each
    // new maximum, so the weights are exp(lse_c - max) with max over all chunks, as above.  (Groups
    // of 8 take 103 registers, of 12 139: the wider form only where it saves a round trip.)
    float mx = -INFINITY, wsum = 0.f, acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    for (int c0 = 0; c0 < S; c0 += kGroup) {
        float lc[kGroup];
        float4 v0[kGroup], v1[kGroup];
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            const int c = c0 + k;
            if (c < S) {
                lc[k] = __ldg(a.part_lse + row0 + c * (2 * BM));
                const float4 *p4 = reinterpret_cast<const float4 *>(a.part_o) +
                                   ((static_cast<int64_t>(local) * S + c) * (D / 4) + 2 * cg) * (2 * BM) + rr;
                v0[k] = __ldg(p4);
                v1[k] = __ldg(p4 + 2 * BM);
            } else {
                lc[k] = -INFINITY;
                v0[k] = v1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float gm = mx;
#pragma unroll
        for (int k = 0; k < kGroup; ++k) gm = fmaxf(gm, lc[k]);
        if (gm == -INFINITY) continue;  // nothing finite yet
        const float sc = mx == -INFINITY ? 0.f : ptx::ex2((mx - gm) * kLog2e);
        wsum *= sc;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] *= sc;
        mx = gm;
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
            const float w = lc[k] == -INFINITY ? 0.f : ptx::ex2((lc[k] - mx) * kLog2e);
            wsum += w;
            acc[0] = fmaf(w, v0[k].x, acc[0]);
            acc[1] = fmaf(w, v0[k].y, acc[1]);
            acc[2] = fmaf(w, v0[k].z, acc[2]);
            acc[3] = fmaf(w, v0[k].w, acc[3]);
            acc[4] = fmaf(w, v1[k].x, acc[4]);
            acc[5] = fmaf(w, v1[k].y, acc[5]);
            acc[6] = fmaf(w, v1[k].z, acc[6]);
            acc[7] = fmaf(w, v1[k].w, acc[7]);
        }
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    uint16_t *dst = a.out + (static_cast<int64_t>(tok) * a.Hq + hq) * D + cg * 8;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(ptx::pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                 ptx::pack_bf16x2(acc[2] * inv, acc[3] * inv),
                                                 ptx::pack_bf16x2(acc[4] * inv, acc[5] * inv),
                                                 ptx::pack_bf16x2(acc[6] * inv, acc[7] * inv));
    if (a.lse && cg == 0) a.lse[static_cast<int64_t>(hq) * a.rows + tok] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
}

}  // namespace
}  // namespace blink

namespace blink {
namespace {

constexpr int kMinSplitTiles = 4;  // prefix tiles a chunk keeps at least

// Very short work runs the single-tile kernel: a block's KV iterations, estimated as the longest
// prefix in tiles plus half the longest tail in tiles (a block's causal span averages half its
// question), at most 8.  Measured: single-tile 6 % faster on 256 causal sequences of 200-1000
// tokens (about 4 iterations a block); the same on a 2048-token prefix (17); 7 % slower on 8
// requests with 2048-token prefixes and 13-14 % slower on 18k and 131k prefixes, where the
// two-tile kernel reads each K/V tile once for 256 rows.
bool use_single_tile(const AttnArgs &a, int max_tail)
{
    int n_pre = 0;
    for (int r = 0; r < a.n_req; ++r) n_pre = max(n_pre, (a.req_P[r] + BN - 1) / BN);
    return n_pre + (max_tail / 2 + BN - 1) / BN <= 8;
}

// Prefix chunks (one request with a prefix).  Launch time is modelled in KV-tile iterations:
// waves(blocks) * (tiles a block runs + kFixedTiles), where a wave is one block per SM, plus,
// when anything is split, the merge launch and the fp32 partials written and read back
// (bytes / kBytesPerTile).  A unit runs n_pre prefix tiles and about t_est tail tiles (its row
// pair's own span).  Cut in S chunks, chunks 0 .. S-2 take c prefix tiles each and the last one
// the remaining n_pre - (S-1) c (0 <= that <= c) and the tail tiles, c chosen so that the longest
// chunk is shortest.  Two forms are weighed against the unsplit launch:
//   - every unit cut into S >= 2 chunks of c >= kMinSplitTiles tiles, within four waves (a small
//     grid: one question against a long prefix);
//   - whole waves of units unsplit, and only the units of the last, partial wave cut into S
//     chunks (c >= 1 tile) that run as one more wave: they start on the SMs the whole units
//     free first (the 2k workload: 168 units on 152 SMs, 152 whole, 16 in 6 chunks of 3 tiles).
// A split is used when it beats the unsplit launch by at least 10 %.  (Measured: one question
// against an 18k prefix 4x faster in 9 chunks; every unit of the 2k workload cut in 2-4 chunks
// 5-40 % slower, which the model rejects.)
struct SplitPlan {
    int64_t unit0;  // units [0, unit0) run whole; units [unit0, units) run in S chunks
    int S, c;       // chunks per split unit and prefix tiles per chunk; S = 1: nothing split
};

SplitPlan choose_split(int64_t units, int n_pre, int t_est, int d, int sms)
{
    constexpr int64_t kFixedTiles = 4;            // block start, pipeline fill and epilogue
    constexpr int64_t kMergeTiles = 2;            // the merge launch
    constexpr int64_t kBytesPerTile = 9ll << 20;  // DRAM bytes moved in one iteration's time
    SplitPlan plan{units, 1, 1 << 30};
    if (units < 1 || sms < 1 || n_pre < 2) return plan;
    auto waves = [&](int64_t u) { return (u + sms - 1) / sms; };
    auto partial_cost = [&](int64_t split_blocks) {  // fp32 O written and read back
        return kMergeTiles + split_blocks * (2 * BM) * d * 8 / kBytesPerTile;
    };
    // Longest chunk (iterations) of s chunks, c >= min_c tiles each (the smallest c of the
    // shortest); -1 if s does not fit.
    auto chunking = [&](int s, int min_c, int &c) -> int64_t {
        const int lo = max(min_c, (n_pre + s - 1) / s), hi = n_pre / (s - 1);
        if (lo > hi) return -1;
        auto len = [&](int cc) {
            const int64_t last = static_cast<int64_t>(n_pre) - static_cast<int64_t>(s - 1) * cc + t_est;
            return last > cc ? last : static_cast<int64_t>(cc);
        };
        c = min(max((n_pre + t_est + s - 1) / s, lo), hi);
        if (c > lo && len(c - 1) <= len(c)) --c;
        return len(c);
    };
    int64_t best = waves(units) * (n_pre + t_est + kFixedTiles) * 9 / 10;  // a split has to win by 10 %
    for (int s = 2; s <= n_pre + 1 && units * s <= 4LL * sms; ++s) {
        int c = 0;
        const int64_t len = chunking(s, kMinSplitTiles, c);
        if (len < 0) continue;
        const int64_t cost = waves(units * s) * (len + kFixedTiles) + partial_cost(units * s);
        if (cost < best) {
            best = cost;
            plan = SplitPlan{0, s, c};
        }
    }
    const int64_t full = units / sms * sms, rest = units - full;
    for (int s = 2; full > 0 && rest > 0 && s <= n_pre + 1 && rest * s <= sms; ++s) {
        int c = 0;
        const int64_t len = chunking(s, 1, c);
        if (len < 0) continue;
        const int64_t cost = full / sms * (n_pre + t_est + kFixedTiles) + (len + kFixedTiles) + partial_cost(rest * s);
        if (cost < best) {
            best = cost;
            plan = SplitPlan{full, s, c};
        }
    }
    return plan;
}

// Tail tiles a unit is assumed to run in the split model: its row pair's own span.
int tail_tiles_estimate(int tpt) { return (2 * tpt + BN - 1) / BN; }

// Workspace after the 256-byte header when the prefix is split: partial LSE [split units][S][2 BM]
// and partial O [split units][S][d / 4][2 BM] (fp32), each region 256-byte aligned.
struct SplitLayout {
    size_t lse, o, total;
};

SplitLayout split_layout(int64_t units, int S, int d)
{
    SplitLayout l{};
    l.lse = kHeaderBytes;
    l.o = l.lse + align_up(static_cast<size_t>(units) * S * 2 * BM * sizeof(float), 256);
    l.total = l.o + align_up(static_cast<size_t>(units) * S * 2 * BM * d * sizeof(float), 256);
    return l;
}

int sm_count_attention()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

// Validates the common arguments, encodes the tensor maps and launches the kernel for the request
// table already filled in `a` (n_req, req_row, req_pre, req_P).  The arena holds arena_slots
// token rows (every request's prefix lives in it).
blink_status launch_attention(AttnArgs &a, const blink_bf16 *q, const blink_bf16 *k_arena, const blink_bf16 *v_arena,
                              int64_t arena_row_stride, int64_t arena_slots, const blink_bf16 *k_tail,
                              const blink_bf16 *v_tail, const int32_t *d_cu_seqlens, const int32_t *d_seq_start,
                              int32_t B, int32_t rows, int32_t max_tail, int32_t Hq, int32_t Hkv, int32_t d,
                              float scale, blink_bf16 *out, float *lse, void *d_ws, size_t ws_bytes,
                              cudaStream_t stream)
{
    if (!q || !k_tail || !v_tail || !d_cu_seqlens || !out || !d_ws) return BLINK_INVALID_ARG;
    if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (d != 64 && d != 128) || rows < 1 || max_tail < 1)
        return BLINK_INVALID_ARG;
    const int g = Hq / Hkv;
    if (g > BM) return BLINK_INVALID_ARG;
    if (B < 1 || B > BLINK_MAX_PLAN_SEQUENCES) return BLINK_OUT_OF_RANGE;
    if (max_tail > BLINK_MAX_INPUT_TOKENS) return BLINK_OUT_OF_RANGE;
    if (a.n_req < 1 || a.n_req > kMaxRequests) return BLINK_OUT_OF_RANGE;
    bool any_prefix = false;
    if (a.req_row[0] != 0 || a.req_row[a.n_req] != rows) return BLINK_INVALID_ARG;
    for (int r = 0; r < a.n_req; ++r) {
        if (a.req_row[r + 1] < a.req_row[r]) return BLINK_INVALID_ARG;
        if (a.req_P[r] < 0 || a.req_P[r] > BLINK_MAX_INPUT_TOKENS) return BLINK_OUT_OF_RANGE;
        if (a.req_P[r] > 0) {
            any_prefix = true;
            if (a.req_pre[r] < 0 || static_cast<int64_t>(a.req_pre[r]) + a.req_P[r] > arena_slots)
                return BLINK_INVALID_ARG;
        } else {
            a.req_pre[r] = 0;
        }
    }
    if (any_prefix) {
        if (!k_arena || !v_arena || arena_slots < 1 || arena_slots > 0x7FFFFFFF) return BLINK_INVALID_ARG;
        if (arena_row_stride < static_cast<int64_t>(Hkv) * d || arena_row_stride % 8 != 0) return BLINK_INVALID_ARG;
        if (!aligned16(k_arena) || !aligned16(v_arena)) return BLINK_INVALID_ARG;
    }
    if (!aligned16(q) || !aligned16(k_tail) || !aligned16(v_tail) || !aligned16(out)) return BLINK_INVALID_ARG;
    if (ws_bytes < blink_attention_workspace(rows, B, 0, Hq, Hkv, d)) return BLINK_WORKSPACE_TOO_SMALL;

    // blocks per request: pairs of M tiles of tpt tokens over the request's own rows
    const int tpt = BM / g;
    int64_t blocks = 0;
    for (int r = 0; r < a.n_req; ++r) {
        a.req_blk[r] = static_cast<int>(blocks);
        const int64_t tiles = (static_cast<int64_t>(a.req_row[r + 1] - a.req_row[r]) + tpt - 1) / tpt;
        blocks += (tiles + 1) / 2;
        if (blocks > 0x7FFFFFFF) return BLINK_OUT_OF_RANGE;
    }
    a.req_blk[a.n_req] = static_cast<int>(blocks);
    if (Hkv > 65535) return BLINK_OUT_OF_RANGE;
    if (blocks == 0) return BLINK_OK;

    CUtensorMap tm_q, tm_kpre, tm_vpre, tm_ktail, tm_vtail;
    const uint64_t e = 2;  // bytes per bf16
    bool ok = encode_tmap_3d_bf16(&tm_q, q, d, Hq, rows, d * e, static_cast<uint64_t>(Hq) * d * e, 64, g, tpt);
    ok = ok && encode_tmap_3d_bf16(&tm_ktail, k_tail, d, Hkv, rows, d * e, static_cast<uint64_t>(Hkv) * d * e, 64,
                                   1, BN);
    ok = ok && encode_tmap_3d_bf16(&tm_vtail, v_tail, d, Hkv, rows, d * e, static_cast<uint64_t>(Hkv) * d * e, 64,
                                   1, BN);
    if (any_prefix) {
        ok = ok && encode_tmap_3d_bf16(&tm_kpre, k_arena, d, Hkv, static_cast<uint64_t>(arena_slots), d * e,
                                       static_cast<uint64_t>(arena_row_stride) * e, 64, 1, BN);
        ok = ok && encode_tmap_3d_bf16(&tm_vpre, v_arena, d, Hkv, static_cast<uint64_t>(arena_slots), d * e,
                                       static_cast<uint64_t>(arena_row_stride) * e, 64, 1, BN);
    } else {
        tm_kpre = tm_ktail;  // never read: no prefix tiles
        tm_vpre = tm_vtail;
    }
    if (!ok) return BLINK_CUDA_ERROR;

    a.cu = d_cu_seqlens;
    a.seq_start = d_seq_start;
    a.out = out;
    a.lse = lse;
    a.err = &static_cast<WorkspaceHeader *>(d_ws)->error;
    a.rows = rows;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.g = g;
    a.tpt = tpt;
    a.max_tail = max_tail;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(d));
    a.scale_log2 = sc * kLog2e;

    // One request's prefix: split it, for a small grid or for the last partial wave of units (if
    // the workspace has the room).
    a.n_split = 1;
    a.split_tiles = 1 << 30;
    a.part_o = nullptr;
    a.part_lse = nullptr;
    a.n_pairs = static_cast<int>(blocks);
    a.unit0 = 0;
    const int64_t units = blocks * Hkv;
    int64_t whole_units = units;  // units run unsplit
    if (a.n_req == 1 && a.req_P[0] > 0) {
        const SplitPlan plan = choose_split(units, (a.req_P[0] + BN - 1) / BN, tail_tiles_estimate(tpt), d,
                                           sm_count_attention());
        if (plan.S > 1) {
            const SplitLayout lay = split_layout(units - plan.unit0, plan.S, d);
            if (ws_bytes >= lay.total) {
                auto *wsb = static_cast<uint8_t *>(d_ws);
                a.n_split = plan.S;
                a.split_tiles = plan.c;
                a.part_lse = reinterpret_cast<float *>(wsb + lay.lse);
                a.part_o = reinterpret_cast<float *>(wsb + lay.o);
                whole_units = plan.unit0;
            }
        }
    }
    if (units * a.n_split > 0x7FFFFFFF) return BLINK_OUT_OF_RANGE;
    // Unsplit launches of short work run the single-tile kernel (two blocks per SM).
    const bool single = a.n_split == 1 && use_single_tile(a, max_tail);
    if (single) {
        int64_t tblocks = 0;
        for (int r = 0; r < a.n_req; ++r) {
            a.req_blk[r] = static_cast<int>(tblocks);
            tblocks += (static_cast<int64_t>(a.req_row[r + 1] - a.req_row[r]) + tpt - 1) / tpt;
            if (tblocks > 0x7FFFFFFF) return BLINK_OUT_OF_RANGE;
        }
        a.req_blk[a.n_req] = static_cast<int>(tblocks);
        const dim3 grid1(static_cast<unsigned>(tblocks), static_cast<unsigned>(Hkv));
        if (d == 128) {
            const int smem = Layout1<128>::kAlloc;
            if (cudaFuncSetAttribute(attention_single_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess)
                return BLINK_CUDA_ERROR;
            attention_single_kernel<128><<<grid1, kThreads1, smem, stream>>>(tm_q, tm_kpre, tm_vpre, tm_ktail, tm_vtail, a);
        } else {
            // at most two blocks per SM: each takes 256 of the 512 tensor-memory columns
            const int smem = Layout1<64>::kAlloc > 80 * 1024 ? Layout1<64>::kAlloc : 80 * 1024;
            if (cudaFuncSetAttribute(attention_single_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess)
                return BLINK_CUDA_ERROR;
            attention_single_kernel<64><<<grid1, kThreads1, smem, stream>>>(tm_q, tm_kpre, tm_vpre, tm_ktail, tm_vtail, a);
        }
        if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
        return BLINK_OK;
    }
    // One launch: the whole units first (one block each), then the split units (n_split blocks
    // each), so the chunks start on the SMs the whole units free first; then the merge.  Each
    // block takes all 512 tensor-memory columns, so one block fits per SM (for d = 64 enough
    // shared memory is reserved to keep it so).
    const int smem = d == 128 ? Layout<128>::kAlloc : (Layout<64>::kAlloc > 120 * 1024 ? Layout<64>::kAlloc : 120 * 1024);
    if (a.n_split == 1) {
        auto kern = d == 128 ? attention_kernel<128, kWholeUnits> : attention_kernel<64, kWholeUnits>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return BLINK_CUDA_ERROR;
        kern<<<static_cast<unsigned>(units), kThreads, smem, stream>>>(tm_q, tm_kpre, tm_vpre, tm_ktail, tm_vtail, a);
        if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
        return BLINK_OK;
    }
    a.unit0 = static_cast<int>(whole_units);
    const int64_t split_units = units - whole_units;
    auto kern = whole_units > 0
                    ? (d == 128 ? attention_kernel<128, kUnitsThenChunks> : attention_kernel<64, kUnitsThenChunks>)
                    : (d == 128 ? attention_kernel<128, kChunksOnly> : attention_kernel<64, kChunksOnly>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return BLINK_CUDA_ERROR;
    kern<<<static_cast<unsigned>(whole_units + split_units * a.n_split), kThreads, smem, stream>>>(
        tm_q, tm_kpre, tm_vpre, tm_ktail, tm_vtail, a);
    if (cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
    // The merge as a programmatic dependent of that launch: its blocks are scheduled while the
    // attention grid drains and start merging as soon as it ends.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(split_units * (2 * BM / kMergeRows)));
    cfg.blockDim = dim3(static_cast<unsigned>(kMergeRows * (d / 8)));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int nb = static_cast<int>(blocks);
    const bool wide = a.n_split > 8;  // 9-12 chunks in one round trip, 13-24 in two
    const cudaError_t me =
        d == 128 ? cudaLaunchKernelEx(&cfg, wide ? split_merge_kernel<128, 12> : split_merge_kernel<128, 8>, a, nb)
                 : cudaLaunchKernelEx(&cfg, wide ? split_merge_kernel<64, 12> : split_merge_kernel<64, 8>, a, nb);
    if (me != cudaSuccess || cudaGetLastError() != cudaSuccess) return BLINK_CUDA_ERROR;
    return BLINK_OK;
}

}  // namespace
}  // namespace blink

extern "C" size_t blink_attention_workspace(int32_t rows, int32_t B, int32_t P, int32_t Hq, int32_t Hkv, int32_t d)
{
    using namespace blink;
    (void)B;
    if (rows < 1 || P < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (d != 64 && d != 128) || Hq / Hkv > BM)
        return kHeaderBytes;
    const int tpt = BM / (Hq / Hkv);
    const int64_t blocks = ((static_cast<int64_t>(rows) + tpt - 1) / tpt + 1) / 2;
    const SplitPlan plan = choose_split(blocks * Hkv, (P + BN - 1) / BN, tail_tiles_estimate(tpt), d, sm_count_attention());
    return plan.S > 1 ? split_layout(blocks * Hkv - plan.unit0, plan.S, d).total : kHeaderBytes;
}

extern "C" blink_status blink_attention_split_plan(int32_t rows, int32_t P, int32_t Hq, int32_t Hkv, int32_t d,
                                                  int32_t sms, int64_t *whole_units, int32_t *chunks,
                                                  int32_t *chunk_tiles)
{
    using namespace blink;
    if (!whole_units || !chunks || !chunk_tiles) return BLINK_INVALID_ARG;
    if (rows < 1 || P < 0 || P > BLINK_MAX_INPUT_TOKENS || Hq < 1 || Hkv < 1 || Hkv > 65535 || Hq % Hkv != 0 ||
        (d != 64 && d != 128) || Hq / Hkv > BM || sms < 1)
        return BLINK_INVALID_ARG;
    const int tpt = BM / (Hq / Hkv);
    const int64_t units = ((static_cast<int64_t>(rows) + tpt - 1) / tpt + 1) / 2 * Hkv;
    const int n_pre = (P + BN - 1) / BN;
    const SplitPlan plan = P > 0 ? choose_split(units, n_pre, tail_tiles_estimate(tpt), d, sms) : SplitPlan{units, 1, 0};
    *whole_units = plan.S > 1 ? plan.unit0 : units;
    *chunks = plan.S;
    *chunk_tiles = plan.S > 1 ? plan.c : n_pre;
    return BLINK_OK;
}

extern "C" blink_status blink_prefix_tail_attention(const blink_bf16 *q, const blink_bf16 *k_pre,
                                                    const blink_bf16 *v_pre, int64_t pre_row_stride,
                                                    const blink_bf16 *k_tail, const blink_bf16 *v_tail,
                                                    const int32_t *d_cu_seqlens, const int32_t *d_seq_start,
                                                    int32_t B, int32_t rows, int32_t P, int32_t max_tail, int32_t Hq,
                                                    int32_t Hkv, int32_t d, float scale, blink_bf16 *out, float *lse,
                                                    void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    using namespace blink;
    if (P < 0) return BLINK_INVALID_ARG;
    if (P > BLINK_MAX_INPUT_TOKENS) return BLINK_OUT_OF_RANGE;
    if (rows < 1) return BLINK_INVALID_ARG;
    AttnArgs a;
    a.n_req = 1;
    a.req_row[0] = 0;
    a.req_row[1] = rows;
    a.req_pre[0] = 0;
    a.req_P[0] = P;
    return launch_attention(a, q, k_pre, v_pre, pre_row_stride, P, k_tail, v_tail, d_cu_seqlens, d_seq_start, B, rows,
                            max_tail, Hq, Hkv, d, scale, out, lse, d_ws, ws_bytes, stream);
}

extern "C" blink_status blink_prefix_tail_attention_multi(
    const blink_bf16 *q, const blink_bf16 *k_arena, const blink_bf16 *v_arena, int64_t arena_row_stride,
    int64_t arena_slots, const blink_bf16 *k_tail, const blink_bf16 *v_tail, const int32_t *d_cu_seqlens,
    const int32_t *d_seq_start, int32_t B, int32_t rows, int32_t n_req, const int32_t *h_req_rows,
    const int32_t *h_req_prefix_start, const int32_t *h_req_prefix_len, int32_t max_tail, int32_t Hq, int32_t Hkv,
    int32_t d, float scale, blink_bf16 *out, float *lse, void *d_ws, size_t ws_bytes, cudaStream_t stream)
{
    using namespace blink;
    if (!h_req_rows || !h_req_prefix_start || !h_req_prefix_len) return BLINK_INVALID_ARG;
    if (n_req < 1 || n_req > kMaxRequests) return BLINK_OUT_OF_RANGE;
    AttnArgs a;
    a.n_req = n_req;
    for (int r = 0; r <= n_req; ++r) a.req_row[r] = h_req_rows[r];
    for (int r = 0; r < n_req; ++r) {
        a.req_pre[r] = h_req_prefix_start[r];
        a.req_P[r] = h_req_prefix_len[r];
    }
    return launch_attention(a, q, k_arena, v_arena, arena_row_stride, arena_slots, k_tail, v_tail, d_cu_seqlens,
                            d_seq_start, B, rows, max_tail, Hq, Hkv, d, scale, out, lse, d_ws, ws_bytes, stream);
}
