// Fused single-launch decode path on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory): shrink and expand in one persistent kernel.
//
// At decode the branch streams adapter weights: every active slot's A and B are
// read once while x and y are small (llama.cpp LoRA adapter page, section
// "为什么低秩增量可以「后加」": decode is bound by memory bandwidth, the cost
// being extra launches and intermediates).  One launch keeps every SM streaming:
//
//   * Tiles are up to 128 sorted positions of one slot.
//   * Shrink items are (tile, slice, 64-column block of k).  An item stages the
//     tile's x rows (M, the tokens) and the slice's A rows (N = r_s); only real
//     rows are copied, and the rows the MMA reads past them only feed
//     accumulator rows or columns nobody reads.  Splitting by slice keeps each
//     unit's partial sums small (the reductions they cost run at a fixed rate
//     per SM) at the price of reading a tile's x rows once per slice, mostly
//     from L2.  Items are weighted by the
//     bytes they move and every CTA takes a contiguous range of equal weight
//     (split-K over k, TensorRT-LLM LoRA serving page, "path 2: split-K
//     tuning"); a CTA's items of one tile form a unit whose partial sums are
//     added into the fp32 accumulator in the workspace (red.global.add.v4.f32),
//     after which the unit adds its item count to the slot's counter (release).
//     The unit that completes a (slot, slice) count converts that slice's sums
//     into bf16 hi + lo parts (x A^T to about 2^-17 relative), clears the fp32
//     rows and marks the slice ready.
//   * Expand units are (tile, slice, 128 output columns), also balanced by bytes,
//     and run transposed: M = the 128 output columns (B rows), N = the tile's
//     tokens, K = the rank (hi, then lo).  A tensor-memory lane is then an output
//     column and all four lane quarters work on every unit however few tokens
//     it has; a thread adds its column of s * D to the tokens' y rows in fp32 and
//     rounds once to bf16.
//   * Rows are gathered through sorted_ids with per-thread 16-byte asynchronous
//     copies (cp.async), four producer warps taking the ring's stages in turn,
//     each waiting only for its own stage's copies before publishing it (one
//     warp sustains about a quarter of an SM's share of HBM bandwidth).
//
// Every CTA issues all its shrink stages before its first expand stage and
// shrink work waits on nothing outside its CTA, so every counter wait ends; the
// launch is cooperative (all CTAs resident) and every wait is still bounded
// (LORA_ERR_TIMEOUT).  The last expand unit of a (slot, slice) resets its
// counters, so every call leaves the workspace as it found it.  Limits (the host
// routes other cases elsewhere): T <= 2048, r_max <= 64, and the tables for S
// slots and T tokens must fit in shared memory next to the stage ring.
#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace lora {

namespace {

constexpr int kTile = 128;                       // tokens per tile
constexpr int kKB = 64;                          // k per item: one 128-byte row
constexpr int kCW = 128;                         // output columns per expand unit (MMA M)
constexpr int kStages = 4;
constexpr int kSlot = 48 * 1024;                 // bytes per ring stage
constexpr int kGuard = 16 * 1024;                // readable bytes behind the ring
constexpr int kProdWarps = 4;                    // warps 1-4: one stage each in flight
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kEpiWarp0 = 1 + kProdWarps;        // first epilogue warp (a multiple of 4 + 1)
constexpr int kEpiThreads = 256;                 // warps 5-12
constexpr int kThreads = 32 + kProdThreads + kEpiThreads;
constexpr int kMaxTokens = 2048;
constexpr int kSmemLimit = 227 * 1024;
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;  // bound on every wait: 200 ms
constexpr int kBarBytes = 1024;                  // barriers and flags, behind the ring
constexpr int kMaxRows = kTile + 256;            // staged rows of a shrink item: tokens + n * r_s
constexpr int kBarEpi = 2;                       // named barriers 2 and 3: the two epilogue groups

struct Args {
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    const int32_t *sorted_ids;
    const int32_t *seg;
    int32_t *shrink_done;  // [S][LORA_MAX_SLICES] per (slot, slice)
    int32_t *expand_done;
    float *acc;            // [n][T][r_max] fp32 partial sums, zero between calls
    uint16_t *xa_hi;       // [n][T][rpw] bf16 parts of the finished sums
    uint16_t *xa_lo;
    int32_t rpw;           // row stride of xa_hi / xa_lo
    int32_t *err;
    int32_t T;
};

__device__ __forceinline__ int32_t round8(int32_t v) { return (v + 7) & ~7; }
__device__ __forceinline__ int32_t round16(int32_t v) { return (v + 15) & ~15; }
__device__ __forceinline__ uint32_t round1k(uint32_t v) { return (v + 1023u) & ~1023u; }

// Rank padding of the expand operands: K = 16, 32, 48 or 64.  Rows of RP*2
// bytes are stored in the widest swizzle that holds them.
__device__ __forceinline__ int32_t rp_of(int32_t r) { return round16(r); }
__device__ __forceinline__ uint32_t rowb_of(int32_t r) {
    const int32_t rp = rp_of(r);
    return rp == 48 ? 128u : static_cast<uint32_t>(rp * 2);  // 48 is held in 64-wide rows
}

__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads: every
// thread gets the same answer, so a group leaves its loops together.
__device__ __forceinline__ bool named_sync_or(int id, int threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(pred ? 1u : 0u), "r"(id), "r"(threads) : "memory");
    return r != 0;
}

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1,%2,%3,%4};" :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t ldg_u16(const uint16_t *p) {
    uint16_t v;
    asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void stg_u16(uint16_t *p, uint32_t v) {
    asm volatile("st.global.u16 [%0], %1;" :: "l"(p), "h"(static_cast<uint16_t>(v)) : "memory");
}

// One bf16 of y (low half of v) + s * d in fp32, rounded once to bf16.
__device__ __forceinline__ uint32_t add_scaled1(uint32_t v, float d, float s) {
    return pack_bf16x2(bf16lo_to_f32(v) + s * d, 0.f) & 0xffffu;
}

// Exclusive scan of data[0..n) by one whole warp; returns the total.
__device__ int32_t warp_exclusive_scan(int32_t *data, int32_t n, int lane) {
    int32_t carry = 0;
    for (int32_t base = 0; base < n; base += 32) {
        const int32_t idx = base + lane;
        const int32_t v = idx < n ? data[idx] : 0;
        int32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t w = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += w;
        }
        if (idx < n) data[idx] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    return carry;
}

// ---------------------------------------------------------------------------
// Work tables (shared memory, built by the prologue)
// ---------------------------------------------------------------------------
struct Tabs {
    const int32_t *seg;    // [S + 1] segment starts (sorted positions)
    const int32_t *rank;   // [S] rank of a usable slot, else 0
    const int32_t *tslot;  // [NT] slot of tile
    const int32_t *tpre;   // [S] exclusive prefix of tiles per slot
    int32_t NT;
};

struct Tile {
    int32_t s, p0, len, r;
};

__device__ __forceinline__ Tile tile_at(const Tabs &tb, int32_t t) {
    Tile ti;
    ti.s = tb.tslot[t];
    const int32_t j = t - tb.tpre[ti.s];
    ti.p0 = tb.seg[ti.s] + j * kTile;
    ti.len = min(kTile, tb.seg[ti.s + 1] - ti.p0);
    ti.r = tb.rank[ti.s];
    return ti;
}

// Last index i in [0, N) with pref[i] <= v (pref ascending).
__device__ __forceinline__ int32_t last_le(const int32_t *pref, int32_t N, int64_t v) {
    int32_t lo = 0, hi = N;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (pref[mid] <= v) lo = mid + 1;
        else hi = mid;
    }
    return lo - 1;
}

// A CTA's share of a list of weighted work pieces: the pieces whose weight
// start lies in [lo, hi), CTA b of G taking lo = ceil(W b / G).  Every tile
// holds P pieces of equal weight (its weight / P).
struct Range {
    int32_t tile, idx;  // current piece: tile and index within the tile
    int64_t hi;
};

__device__ __forceinline__ Range first_piece(const int32_t *pref, int32_t NT, int32_t P) {
    Range r;
    const int64_t W = pref[NT];
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t lo = (W * b + G - 1) / G;
    r.hi = (W * (b + 1) + G - 1) / G;
    r.tile = NT;
    r.idx = 0;
    if (lo >= W) return r;
    int32_t t = last_le(pref, NT, lo);
    const int32_t w = (pref[t + 1] - pref[t]) / P;
    int32_t i = static_cast<int32_t>((lo - pref[t] + w - 1) / w);
    if (i >= P) {
        ++t;
        i = 0;
    }
    r.tile = t;
    r.idx = i;
    return r;
}

// True while the current piece starts below this CTA's bound.
__device__ __forceinline__ bool piece_valid(const Range &r, const int32_t *pref, int32_t NT, int32_t P) {
    if (r.tile >= NT) return false;
    const int32_t w = (pref[r.tile + 1] - pref[r.tile]) / P;
    return static_cast<int64_t>(pref[r.tile]) + static_cast<int64_t>(r.idx) * w < r.hi;
}

// Number of this CTA's pieces in tile r.tile from r.idx on.
__device__ __forceinline__ int32_t pieces_left_in_tile(const Range &r, const int32_t *pref, int32_t P) {
    const int32_t w = (pref[r.tile + 1] - pref[r.tile]) / P;
    const int64_t room = r.hi - pref[r.tile] - static_cast<int64_t>(r.idx) * w;  // > 0
    const int32_t fit = static_cast<int32_t>((room + w - 1) / w);
    return min(P - r.idx, fit);
}

// Shrink stage: KB items of one (tile, slice), each [x rows N8 | A rows r] x 128 bytes.
__device__ __forceinline__ int32_t shrink_kb_per_stage(int32_t N8, int32_t r) {
    return max(1, kSlot / ((N8 + r) * 128));
}

// Expand: kCW-column chunks of a tile over the slices.
__device__ __forceinline__ int32_t chunks_per_tile(const Shape &sh) {
    int32_t c = 0;
    for (int i = 0; i < sh.n; ++i) c += (sh.off[i + 1] - sh.off[i] + kCW - 1) / kCW;
    return c;
}

__device__ __forceinline__ void chunk_at(const Shape &sh, int32_t c, int32_t &i, int32_t &c0, int32_t &width) {
    i = 0;
    while (true) {
        const int32_t d = sh.off[i + 1] - sh.off[i], nc = (d + kCW - 1) / kCW;
        if (c < nc || i + 1 >= sh.n) {
            c0 = c * kCW;
            width = min(kCW, d - c0);
            return;
        }
        c -= nc;
        ++i;
    }
}

// Records a failure once and tells the other roles to stop.
__device__ __forceinline__ void give_up(int32_t *err, volatile int32_t *abort_flag, int32_t code) {
    report_error(err, code);
    *abort_flag = 1;
}

// ---------------------------------------------------------------------------
// Kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) fused_tc_kernel(Args a, Shape sh, const void *table) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int32_t S = sh.S, T = a.T;
    const int32_t NTmax = S + (T + kTile - 1) / kTile;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kSlot);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint64_t *s_rows = reinterpret_cast<uint64_t *>(smem + kStages * kSlot + kBarBytes);  // [kProdWarps][kMaxRows]
    int32_t *misc = reinterpret_cast<int32_t *>(s_rows + kProdWarps * kMaxRows);  // [8]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
    volatile int32_t *abort_flag = misc + 1;
    int32_t *s_nt = misc + 2;
    volatile int32_t *s_fin = misc + 3;        // [2]: the group's unit completed its slot
    int32_t *s_seg = misc + 8;                 // [S + 1]
    int32_t *s_rank = s_seg + S + 1;           // [S]
    int32_t *s_tpre = s_rank + S;              // [S]
    int32_t *s_tslot = s_tpre + S;             // [NTmax]
    int32_t *s_tsh = s_tslot + NTmax;          // [NTmax + 1]
    int32_t *s_tex = s_tsh + NTmax + 1;        // [NTmax + 1]
    int32_t *s_ready = s_tex + NTmax + 1;      // [S] bit i: slice i of the slot seen ready
    int32_t *s_tok = s_ready + S;              // [T]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TableView tab(table, sh.S, sh.n);
    const int32_t nkb = (sh.k + kKB - 1) / kKB;
    const int32_t P_sh = sh.n * nkb;  // shrink items per tile: slices x blocks of k
    const int32_t C = chunks_per_tile(sh);

    // ------------------------------------------------------------ prologue
    // Loads that do not depend on the table header go out first; warp 0 reads
    // the ranks once the header shows the table holds S slots and builds the
    // work tables with shuffle scans, while the other warps wait.
    const int32_t *hdr = static_cast<const int32_t *>(table);
    const bool ok = hdr[0] == kTableMagic && hdr[1] == S && hdr[2] == sh.n && a.seg[S + 1] == T;
    for (int t = tid; t < T; t += kThreads) {
        int32_t v = a.sorted_ids[t];
        if (v < 0 || v >= T) {
            report_error(a.err, LORA_ERR_INVALID_ARG);
            v = -1;
        }
        s_tok[t] = v;
    }
    for (int s = tid; s <= S; s += kThreads) s_seg[s] = a.seg[s];
    if (warp == 0) {
        if (!ok && lane == 0 && blockIdx.x == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
        for (int s = lane; s < S; s += 32) {
            const int32_t r = ok ? tab.rank[s] : 0;
            const int32_t cnt = ok ? a.seg[s + 1] - a.seg[s] : 0;
            if (r > sh.r_max && blockIdx.x == 0) report_error(a.err, LORA_ERR_RANK);
            const bool use = ok && cnt > 0 && r > 0 && r <= sh.r_max;
            s_rank[s] = use ? r : 0;
            s_tpre[s] = use ? (cnt + kTile - 1) / kTile : 0;
            s_ready[s] = 0;
        }
        __syncwarp();
        const int32_t NT = warp_exclusive_scan(s_tpre, S, lane);
        for (int s = lane; s < S; s += 32) {
            const int32_t r = s_rank[s];
            if (r == 0) continue;
            const int32_t cnt = a.seg[s + 1] - a.seg[s], tiles = (cnt + kTile - 1) / kTile;
            const int32_t rp = rp_of(r);
            for (int j = 0; j < tiles; ++j) {
                const int32_t t = s_tpre[s] + j, len = min(kTile, cnt - j * kTile);
                s_tslot[t] = s;
                s_tsh[t] = sh.n * nkb * (round8(len) + r);  // 128-byte rows: items x (tokens + A rows)
                s_tex[t] = C * (2 * rp + 4 * len + 8);    // per unit: B rows, y in and out, fixed cost
            }
        }
        __syncwarp();
        const int32_t Wsh = warp_exclusive_scan(s_tsh, NT, lane);
        const int32_t Wex = warp_exclusive_scan(s_tex, NT, lane);
        if (lane == 0) {
            s_tsh[NT] = Wsh;
            s_tex[NT] = Wex;
            *s_nt = NT;
            *abort_flag = 0;
            for (int st = 0; st < kStages; ++st) {
                tc::mbar_init(&full[st], 32);  // the publishing warp
                tc::mbar_init(&empty[st], 1);
            }
            for (int b = 0; b < 2; ++b) {
                tc::mbar_init(&acc_full[b], 1);
                tc::mbar_init(&acc_empty[b], 1);
            }
            tc::mbar_init(drain, 1);
            tc::mbar_init_fence();
        }
        __syncwarp();
        tc::tmem_alloc(tmem_slot, 512);
        tc::fence_before_sync();
    } else if (warp < kEpiWarp0 && ok) {
        // while warp 0 builds the tables, pull the table's weight pointers into L1
        // (the producers read them for every unit)
        for (int e = tid - 32; e < S * sh.n; e += kProdThreads) {
            uint64_t pa, pb;
            asm volatile("ld.global.u64 %0, [%1];" : "=l"(pa) : "l"(tab.a_ptr + e));
            asm volatile("ld.global.u64 %0, [%1];" : "=l"(pb) : "l"(tab.b_ptr + e));
        }
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = tc::smem_u32(smem);
    const int32_t NT = *s_nt;

    Tabs tb;
    tb.seg = s_seg;
    tb.rank = s_rank;
    tb.tslot = s_tslot;
    tb.tpre = s_tpre;
    tb.NT = NT;

    if (warp == 0) {
        // ================================================== MMA issuer
        if (lane == 0) {
            int32_t it = 0, u = 0;
            bool stop = false;
            // shrink units: D[token, rank] += x A_i^T for one slice per unit
            Range rg = first_piece(s_tsh, NT, P_sh);
            while (!stop && piece_valid(rg, s_tsh, NT, P_sh)) {
                const Tile ti = tile_at(tb, rg.tile);
                const int32_t kb0 = rg.idx % nkb;
                const int32_t nitems = min(pieces_left_in_tile(rg, s_tsh, P_sh), nkb - kb0);
                const int32_t N8 = round8(ti.len), kbs = shrink_kb_per_stage(N8, ti.r);
                const uint32_t idesc = tc::idesc_bf16(kTile, round16(ti.r));
                const int32_t b = u & 1;
                if (u >= 2 && !tc::mbar_wait(&acc_empty[b], ((u >> 1) - 1) & 1, abort_flag, kWaitNs)) {
                    give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                    break;
                }
                tc::fence_after_sync();
                for (int32_t q = 0; q < nitems; q += kbs, ++it) {
                    const int st = it % kStages;
                    if (!tc::mbar_wait(&full[st], (it / kStages) & 1, abort_flag, kWaitNs)) {
                        give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                        stop = true;
                        break;
                    }
                    tc::fence_after_sync();
                    const int32_t m = min(kbs, nitems - q);
                    for (int32_t e = 0; e < m; ++e) {
                        const uint32_t xs = sbase + st * kSlot + e * (N8 + ti.r) * 128;
                        const uint32_t as = xs + N8 * 128;
#pragma unroll
                        for (int kk = 0; kk < kKB / 16; ++kk)
                            tc::mma_bf16(tmem + b * 256, tc::smem_desc(xs + 32 * kk, 1024, tc::kLayoutSW128),
                                         tc::smem_desc(as + 32 * kk, 1024, tc::kLayoutSW128), idesc,
                                         q + e + kk > 0);
                    }
                    tc::mma_commit(&empty[st]);
                }
                if (stop) break;
                tc::mma_commit(&acc_full[b]);
                ++u;
                rg.idx += nitems;
                if (rg.idx >= P_sh) {
                    ++rg.tile;
                    rg.idx = 0;
                }
            }
            // expand units, transposed: D[column, token] = B xa_hi^T + B xa_lo^T
            Range re = first_piece(s_tex, NT, C);
            while (!stop && piece_valid(re, s_tex, NT, C)) {
                const Tile ti = tile_at(tb, re.tile);
                const uint32_t rowb = rowb_of(ti.r);
                const uint32_t layout = tc::layout_for_rowb(rowb);
                const int32_t N16 = round16(ti.len);
                const uint32_t bsz = kCW * rowb, xsz = round1k(static_cast<uint32_t>(N16) * rowb);
                const uint32_t idesc = tc::idesc_bf16(kCW, N16);
                const int32_t b = u & 1;
                const int st = it % kStages;
                if ((u >= 2 && !tc::mbar_wait(&acc_empty[b], ((u >> 1) - 1) & 1, abort_flag, kWaitNs)) ||
                    !tc::mbar_wait(&full[st], (it / kStages) & 1, abort_flag, kWaitNs)) {
                    give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t ob = sbase + st * kSlot;
                const int32_t ksteps = rp_of(ti.r) / 16;
                for (int kk = 0; kk < ksteps; ++kk) {
                    // K steps of 16 within a swizzled row: +32 bytes
                    const uint64_t ad = tc::smem_desc(ob + 32 * kk, 8 * rowb, layout);
                    tc::mma_bf16(tmem + b * 256, ad, tc::smem_desc(ob + bsz + 32 * kk, 8 * rowb, layout), idesc, kk > 0);
                    tc::mma_bf16(tmem + b * 256, ad, tc::smem_desc(ob + bsz + xsz + 32 * kk, 8 * rowb, layout), idesc,
                                 true);
                }
                tc::mma_commit(&empty[st]);
                tc::mma_commit(&acc_full[b]);
                ++it;
                ++u;
                if (++re.idx >= C) {
                    ++re.tile;
                    re.idx = 0;
                }
            }
            tc::mma_commit(drain);
            if (!tc::mbar_wait_timed(drain, 0, kWaitNs)) report_error(a.err, LORA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        // ================================================== producers
        // The warps take the stages in turn (stage it belongs to warp
        // it % kProdWarps).  A warp issues its stage's copies, waits for its own
        // copies only, makes them visible to the tensor cores and publishes the
        // stage: every stage of the ring is in flight and none waits for a later
        // one to be issued.
        const int pw = warp - 1;
        int32_t it = 0;           // global stage index
        bool stop = false;
        int32_t pend_slot = -1, pend_old = 0, pend_total = 0;  // this lane's deferred count: (slot, slice)
        auto wait_slot_free = [&](int32_t st_it) -> bool {
            if (st_it < kStages) return true;
            return __all_sync(0xffffffffu, tc::mbar_wait(&empty[st_it % kStages], ((st_it / kStages) - 1) & 1,
                                                           abort_flag, kWaitNs));
        };
        auto publish = [&](int32_t st_it) {
            tc::cp_wait_all();
            tc::fence_async_smem();
            tc::mbar_arrive(&full[st_it % kStages]);
        };
        // ---- shrink stages
        Range rg = first_piece(s_tsh, NT, P_sh);
        while (!stop && piece_valid(rg, s_tsh, NT, P_sh)) {
            const Tile ti = tile_at(tb, rg.tile);
            const int32_t kb0 = rg.idx % nkb, slice = rg.idx / nkb;
            const int32_t nitems = min(pieces_left_in_tile(rg, s_tsh, P_sh), nkb - kb0);
            const int32_t N8 = round8(ti.len), kbs = shrink_kb_per_stage(N8, ti.r);
            const int c = lane & 7, r0 = lane >> 3;  // this lane's 16-byte column and first row
            const int32_t rows = ti.len + ti.r;
            // this warp's row table for the unit: address of each staged row's
            // element 0 (0 = a token out of range: the row reads as zero); token rows
            // first, then the slice's A rows
            uint64_t *tbl = s_rows + pw * kMaxRows;
            __syncwarp();
            const uint64_t abase = tab.a_ptr[ti.s * sh.n + slice];
            for (int32_t row = lane; row < rows; row += 32) {
                uint64_t src;
                if (row < ti.len) {
                    const int32_t t = s_tok[ti.p0 + row];
                    src = t >= 0 ? reinterpret_cast<uint64_t>(a.x + static_cast<int64_t>(t) * a.ldx) : 0;
                } else {
                    src = abase + static_cast<uint64_t>(row - ti.len) * sh.k * 2;
                }
                tbl[row] = src;
            }
            __syncwarp();
            for (int32_t q = 0; q < nitems; q += kbs, ++it) {
                if (it % kProdWarps != pw) continue;
                if (!wait_slot_free(it)) {
                    give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                    stop = true;
                    break;
                }
                const uint32_t sb = sbase + (it % kStages) * kSlot;
                const int32_t m = min(kbs, nitems - q);
                for (int32_t e = 0; e < m; ++e) {
                    const int32_t col = (kb0 + q + e) * kKB + 8 * c;
                    const bool inb = col < sh.k;
                    const uint32_t ib = sb + e * (N8 + ti.r) * 128;
#pragma unroll 4
                    for (int32_t row = r0; row < rows; row += 4) {
                        const uint64_t src = tbl[row];
                        const int32_t d = row < ti.len ? row : row - ti.len + N8;
                        const bool v = inb && src != 0;
                        tc::cp16(ib + d * 128 + ((c ^ (d & 7)) << 4),
                                 v ? reinterpret_cast<const void *>(src + 2 * static_cast<uint64_t>(col)) : a.x, v);
                    }
                }
                publish(it);
            }
            rg.idx += nitems;
            if (rg.idx >= P_sh) {
                ++rg.tile;
                rg.idx = 0;
            }
        }
        // ---- expand stages: B rows of the chunk, then the tile's xa hi/lo rows
        int32_t my_exp = 0;  // expand stages of this warp so far
        Range re = first_piece(s_tex, NT, C);
        while (!stop && piece_valid(re, s_tex, NT, C)) {
            const Tile ti = tile_at(tb, re.tile);
            const int32_t this_it = it++, this_c = re.idx;
            if (++re.idx >= C) {
                ++re.tile;
                re.idx = 0;
            }
            if (this_it % kProdWarps != pw) continue;
            int32_t i, c0, width;
            chunk_at(sh, this_c, i, c0, width);
            const int32_t rp = rp_of(ti.r);
            const uint32_t rowb = rowb_of(ti.r), cpr_log = rowb == 128 ? 3u : (rowb == 64 ? 2u : 1u);
            const uint32_t bsz = kCW * rowb, xsz = round1k(static_cast<uint32_t>(round16(ti.len)) * rowb);
            if (!wait_slot_free(this_it)) {
                give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                stop = true;
                break;
            }
            const uint32_t ob = sbase + (this_it % kStages) * kSlot;
            // B rows (output columns) of the chunk; ranks j >= r_s read as zero
            const uint16_t *B = reinterpret_cast<const uint16_t *>(tab.b_ptr[ti.s * sh.n + i]);
            for (int32_t z = lane; z < (width << cpr_log); z += 32) {
                const int32_t m = z >> cpr_log, cc = z & ((1 << cpr_log) - 1);
                const bool v = 8 * cc < ti.r;
                tc::cp16(ob + tc::swz_offset(m, cc, rowb), v ? B + static_cast<int64_t>(c0 + m) * ti.r + 8 * cc : a.x, v);
            }
            // the slice is ready once its counter passed every item plus the conversion
            const int32_t tiles_s = (s_seg[ti.s + 1] - s_seg[ti.s] + kTile - 1) / kTile;
            const int32_t si = ti.s * LORA_MAX_SLICES + i;
            if (lane == 0 && !((s_ready[ti.s] >> i) & 1)) {
                const int32_t need = tiles_s * nkb + 1;
                const uint64_t t0 = globaltimer_ns();
                int spin = 0;
                while (ld_acquire(&a.shrink_done[si]) < need) {
                    __nanosleep(200);  // poll gently: the other warps are streaming
                    if ((++spin & 15) == 0 && (globaltimer_ns() - t0 > kWaitNs || *abort_flag)) {
                        give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                        break;
                    }
                }
                atomicOr(&s_ready[ti.s], 1 << i);
            }
            __syncwarp();
            if (__any_sync(0xffffffffu, *abort_flag != 0)) {
                stop = true;
                break;
            }
            // the tile's x A^T rows of slice i as bf16 hi and lo (chunks past rp are never read)
            const size_t hl_row = static_cast<size_t>(i) * T;
            for (int32_t z = lane; z < (ti.len << cpr_log); z += 32) {
                const int32_t row = z >> cpr_log, cc = z & ((1 << cpr_log) - 1);
                if (8 * cc >= rp) continue;
                const int32_t t = s_tok[ti.p0 + row];
                const bool v = t >= 0;
                const size_t o = (hl_row + (v ? t : 0)) * a.rpw + 8 * cc;
                const uint32_t d = tc::swz_offset(row, cc, rowb);
                tc::cp16(ob + bsz + d, a.xa_hi + o, v);
                tc::cp16(ob + bsz + xsz + d, a.xa_lo + o, v);
            }
            // count this unit's read of the slot; the result is looked at after the
            // loop, where the last reader of a slot resets its counters
            if (lane == (my_exp & 31)) {
                if (pend_slot >= 0 && pend_old == pend_total - 1) {  // a second count on this lane: settle the first
                    a.shrink_done[pend_slot] = 0;
                    a.expand_done[pend_slot] = 0;
                }
                pend_slot = si;
                pend_total = tiles_s * ((sh.off[i + 1] - sh.off[i] + kCW - 1) / kCW);
                pend_old = atomicAdd(&a.expand_done[si], 1);
            }
            ++my_exp;
            publish(this_it);
        }
        tc::cp_wait_all();
        if (pend_slot >= 0 && pend_old == pend_total - 1) {
            a.shrink_done[pend_slot] = 0;
            a.expand_done[pend_slot] = 0;
        }
    } else {
        // ================================================== epilogue
        // Two groups of four warps take alternate units (and so the two
        // accumulators), so one unit's memory latency overlaps the other's; warp q
        // of a group reads tensor-memory lanes 32q..32q+31.
        const int ew = warp - kEpiWarp0, q = warp & 3, grp = ew >> 2;
        const int bar_id = kBarEpi + grp;
        const int gt = 32 * q + lane;  // 0..127: this thread's tensor-memory lane
        int32_t u = 0;
        bool stop = false;
        // ---- shrink units: partial sums -> fp32 accumulator rows (lane = token)
        Range rg = first_piece(s_tsh, NT, P_sh);
        while (!stop && piece_valid(rg, s_tsh, NT, P_sh)) {
            const Tile ti = tile_at(tb, rg.tile);
            const int32_t kb0 = rg.idx % nkb, slice = rg.idx / nkb;
            const int32_t nitems = min(pieces_left_in_tile(rg, s_tsh, P_sh), nkb - kb0);
            const int32_t b = u & 1;
            const int32_t this_u = u++;
            rg.idx += nitems;
            if (rg.idx >= P_sh) {
                ++rg.tile;
                rg.idx = 0;
            }
            if (b != grp) continue;
            bool fail = !__all_sync(0xffffffffu, tc::mbar_wait(&acc_full[b], (this_u >> 1) & 1, abort_flag, kWaitNs));
            if (fail) give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
            tc::fence_after_sync();
            if (!fail && 32 * q < ti.len) {
                const int32_t t = gt < ti.len ? s_tok[ti.p0 + gt] : -1;
                uint32_t v[64];
                const int32_t R16 = round16(ti.r);
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    if (16 * h < R16)
                        tc::tmem_ld16_async(tmem + (static_cast<uint32_t>(32 * q) << 16) + b * 256 + 16 * h, v + 16 * h);
                tc::tmem_wait_ld64(v);
                if (t >= 0) {
                    float *dst = a.acc + (static_cast<int64_t>(slice) * T + t) * sh.r_max;
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (4 * e < ti.r)
                            red_add_v4(dst + 4 * e, __uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                       __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                }
            }
            tc::fence_before_sync();
            stop = named_sync_or(bar_id, 128, fail || *abort_flag);
            const int32_t need = ((s_seg[ti.s + 1] - s_seg[ti.s] + kTile - 1) / kTile) * nkb;
            int32_t *cnt_si = a.shrink_done + ti.s * LORA_MAX_SLICES + slice;
            if (gt == 0) {
                tc::mbar_arrive(&acc_empty[b]);
                s_fin[grp] = 0;
                if (!stop) {
                    // the barrier ordered the group's reductions before this GPU-scope
                    // fence, which releases them with the count; the fence after the
                    // add makes the other units' sums visible to a finishing group
                    __threadfence();
                    const int32_t old = atomicAdd(cnt_si, nitems);
                    __threadfence();
                    s_fin[grp] = old + nitems == need;
                }
            }
            named_sync(bar_id, 128);
            if (s_fin[grp]) {
                // the slice's sums are final: bf16 hi + lo for the expand, fp32 rows cleared
                const int32_t p0 = s_seg[ti.s], cnt = s_seg[ti.s + 1] - p0, rp = rp_of(ti.r), g4 = rp / 4;
                const int32_t total = cnt * g4;
                // five independent loads in flight per thread; the index arithmetic
                // is redone for the stores rather than kept in registers
                for (int32_t z0 = gt; z0 < total; z0 += 128 * 5) {
                    float4 v[5];
#pragma unroll
                    for (int u8 = 0; u8 < 5; ++u8) {
                        const int32_t z = z0 + 128 * u8;
                        v[u8] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (z < total) {
                            const int32_t row = z / g4, j = 4 * (z - row * g4), t = s_tok[p0 + row];
                            if (t >= 0 && j < ti.r)
                                v[u8] = ldg_cg_f4(a.acc + (static_cast<int64_t>(slice) * T + t) * sh.r_max + j);
                        }
                    }
#pragma unroll
                    for (int u8 = 0; u8 < 5; ++u8) {
                        const int32_t z = z0 + 128 * u8;
                        if (z >= total) continue;
                        const int32_t row = z / g4, j = 4 * (z - row * g4), t = s_tok[p0 + row];
                        if (t < 0) continue;
                        const int64_t rowi = static_cast<int64_t>(slice) * T + t;
                        if (j < ti.r)
                            *reinterpret_cast<float4 *>(a.acc + rowi * sh.r_max + j) = make_float4(0.f, 0.f, 0.f, 0.f);
                        uint32_t h0, l0, h1, l1;
                        split_bf16x2(v[u8].x, v[u8].y, h0, l0);
                        split_bf16x2(v[u8].z, v[u8].w, h1, l1);
                        const size_t o = static_cast<size_t>(rowi) * a.rpw + j;
                        *reinterpret_cast<uint2 *>(a.xa_hi + o) = make_uint2(h0, h1);
                        *reinterpret_cast<uint2 *>(a.xa_lo + o) = make_uint2(l0, l1);
                    }
                }
                named_sync(bar_id, 128);
                if (gt == 0) {
                    __threadfence();
                    atomicAdd(cnt_si, 1);  // ready
                }
            }
        }
        // ---- expand units: y[token, column] += s * D[column, token] (lane = column)
        Range re = first_piece(s_tex, NT, C);
        while (!stop && piece_valid(re, s_tex, NT, C)) {
            const Tile ti = tile_at(tb, re.tile);
            const int32_t this_u = u++, this_c = re.idx, b = this_u & 1;
            if (++re.idx >= C) {
                ++re.tile;
                re.idx = 0;
            }
            if (b != grp) continue;
            int32_t i, c0, width;
            chunk_at(sh, this_c, i, c0, width);
            const float sc = tab.scale[ti.s];
            const bool colv = gt < width;
            uint16_t *ycol = a.y + sh.off[i] + c0 + gt;
            // 32 tokens per step: this column's y values of the next 32 tokens are
            // in flight while the current ones are added and stored
            auto load_y = [&](int32_t t0, uint32_t (&dst)[32]) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int32_t tt = t0 + e;
                    const int32_t t = tt < ti.len ? s_tok[ti.p0 + tt] : -1;
                    dst[e] = (colv && t >= 0) ? ldg_u16(ycol + static_cast<int64_t>(t) * a.ldy) : 0u;
                }
            };
            uint32_t yv[32];
            load_y(0, yv);
            bool fail = !__all_sync(0xffffffffu, tc::mbar_wait(&acc_full[b], (this_u >> 1) & 1, abort_flag, kWaitNs));
            if (fail) give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
            tc::fence_after_sync();
            if (!fail) {
                const int32_t N16 = round16(ti.len);
                for (int32_t t0 = 0; t0 < ti.len; t0 += 32) {
                    uint32_t v[32];
                    tc::tmem_ld16_async(tmem + (static_cast<uint32_t>(32 * q) << 16) + b * 256 + t0, v);
                    if (t0 + 16 < N16)
                        tc::tmem_ld16_async(tmem + (static_cast<uint32_t>(32 * q) << 16) + b * 256 + t0 + 16, v + 16);
                    tc::tmem_wait_ld32(v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = add_scaled1(yv[e], __uint_as_float(v[e]), sc);
                    if (t0 + 32 < ti.len) load_y(t0 + 32, yv);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int32_t tt = t0 + e;
                        const int32_t t = tt < ti.len ? s_tok[ti.p0 + tt] : -1;
                        if (colv && t >= 0) stg_u16(ycol + static_cast<int64_t>(t) * a.ldy, v[e]);
                    }
                }
            }
            tc::fence_before_sync();
            stop = named_sync_or(bar_id, 128, fail || *abort_flag);
            if (gt == 0) tc::mbar_arrive(&acc_empty[b]);
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

size_t fused_tc_smem(int32_t S, int32_t T) {
    const size_t NTmax = static_cast<size_t>(S) + (T + kTile - 1) / kTile;
    const size_t tables =
        kBarBytes + 8 * kProdWarps * kMaxRows + 4 * (8 + (S + 1) + 2 * S + NTmax + 2 * (NTmax + 1) + S + T);
    return 1024 + static_cast<size_t>(kStages) * kSlot + std::max<size_t>(tables, kGuard);
}

}  // namespace

bool fused_tc_supported(int32_t T, const Shape &sh) {
    // the work weights are summed in int32: bound d and k well below overflow;
    // the tables for S slots and T tokens must fit next to the stage ring
    return T <= kMaxTokens && sh.r_max <= 64 && sh.off[sh.n] <= 65536 && sh.k <= 65536 &&
           fused_tc_smem(sh.S, T) <= static_cast<size_t>(kSmemLimit);
}

cudaError_t launch_fused_tc(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                            const void *table, const int32_t *sorted_ids, const int32_t *seg, float *ws, int32_t T,
                            int32_t *err, cudaStream_t stream) {
    static int num_sms = 0;
    static bool attr_set = false;
    if (!fused_tc_supported(T, sh)) return cudaErrorNotSupported;
    if (!attr_set) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(fused_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_tc_kernel, kThreads, kSmemLimit);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        attr_set = true;
    }
    const WorkspaceLayout L(T, sh.n, sh.r_max, sh.S);
    char *base = reinterpret_cast<char *>(ws);
    Args a;
    a.x = x;
    a.ldx = ldx;
    a.y = y;
    a.ldy = ldy;
    a.sorted_ids = sorted_ids;
    a.seg = seg;
    a.shrink_done = reinterpret_cast<int32_t *>(base);
    a.expand_done = a.shrink_done + static_cast<size_t>(sh.S) * LORA_MAX_SLICES;
    a.acc = reinterpret_cast<float *>(base + L.acc_off);
    a.xa_hi = reinterpret_cast<uint16_t *>(base + L.hi_off);
    a.xa_lo = reinterpret_cast<uint16_t *>(base + L.lo_off);
    a.rpw = tc_rank_pad(sh.r_max);
    a.err = err;
    a.T = T;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = fused_tc_smem(sh.S, T);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_tc_kernel, a, sh, table);
}

}  // namespace lora
