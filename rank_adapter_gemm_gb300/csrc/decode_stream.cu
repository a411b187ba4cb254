// Decode-size LoRA branch as two streaming kernels on warp-level tensor-core
// MMA (mma.sync m16n8k16, bf16 in, fp32 accumulate).
//
// At decode the branch streams adapter weights: every active slot's A and B are
// read once while x and y are small (llama.cpp LoRA adapter page, section
// "为什么低秩增量可以「后加」": decode is bound by memory bandwidth, the cost
// being extra launches and intermediates).  So both kernels are built around
// keeping HBM busy from the first microsecond to the last:
//
//   * Work is a list of tiles (up to 64 sorted positions of one slot for the
//     shrink, 32 for the expand), each cut into pieces of equal bytes: shrink
//     pieces are (slice, rank group of <= 64 rows, 64 columns of k), expand
//     pieces (slice, 32 output columns).  CTA b of G takes the pieces whose
//     byte offset lies in [W b / G, W (b + 1) / G): every SM moves the same
//     bytes, and big slots are split over k across SMs (split-K, TensorRT-LLM
//     LoRA serving page, "path 2: split-K tuning").  A CTA's consecutive
//     pieces of one (tile, slice, rank group) form a unit.
//   * Four producer warps gather the rows (A rows and the tiles' token rows of
//     x; B rows, y rows and accumulator rows) with 16-byte asynchronous copies
//     (cp.async), each lane signalling the stage's mbarrier when its copies
//     land (cp.async.mbarrier.arrive.noinc), so a producer never waits for its
//     own data and the ring stays full.  Bulk (TMA) copies are not used here:
//     one row per copy leaves the copy engine issue-bound far below HBM speed.
//     Four consumer warps read the stages with ldmatrix (shrink rows in 128-byte
//     lines with the 16-byte chunks XOR-swizzled by row, other rows at a pitch
//     of 16 mod 128 bytes: no bank conflicts).
//   * The shrink keeps each warp's partial sums in registers across the stages
//     of a unit and adds them into an fp32 accumulator in the workspace once
//     per unit (red.global.add.v4.f32).
//   * The expand is launched as a programmatic dependent of the shrink, and the
//     two are sized so that one CTA of each fits on an SM (shared memory,
//     and 4 warps x 128 registers on each SM sub-partition): while the shrink
//     streams A, the expand's CTAs build their tables, clear their share of the
//     other accumulator buffer and copy their first stages of B and y; only the
//     accumulator rows wait for the shrink grid (griddepcontrol.wait).  The
//     sums enter the MMA as bf16 hi + lo parts (x A^T to about 2^-17 relative);
//     y = bf16(y + s * xa B^T) with one rounding.
//   * The workspace holds two accumulator buffers and a call counter g: a call
//     adds into buffer g & 1 and clears buffer (g + 1) & 1, which the previous
//     call used; the expand's last CTA advances g.  No CTA waits on another.
//
// Limits (the host routes other cases elsewhere): T <= 2048, r_max <= 128,
// k % 16 == 0, k <= 65536, sum of slice widths <= 65536, and the tables for S
// slots and T tokens must fit in shared memory next to the ring.
#include <algorithm>

#include "common.cuh"
#include "schedule.cuh"

namespace lora {

namespace {

// Both kernels: warps 0-3 consume, warps 4-7 produce.  One CTA of each shares
// an SM: 16 warps, 4 on each sub-partition, at 128 registers a thread.
constexpr int kCWarps = 4;
constexpr int kPWarps = 4;
constexpr int kThreads = 32 * (kCWarps + kPWarps);
constexpr int kSStages = 6;                     // shrink ring
constexpr int kSSlot = 16 * 1024;
constexpr int kEStages = 4;                     // expand ring
constexpr int kESlot = 24 * 1024;
// Stage it is filled by producer warp it % kPWarps once the consumers have
// released stage it - stages.  With at least as many stages as producer warps,
// a warp's previous wait already saw the release of stage it - 2 * stages, so
// the phase parity it waits for cannot alias an older phase.
static_assert(kSStages >= kPWarps && kEStages >= kPWarps, "ring shallower than the producer rotation");
constexpr int kTG = 64;                         // shrink tile: tokens
constexpr int kTGe = 32;                        // expand tile: tokens (16 for ranks above 64)
constexpr int kRG = 64;                         // shrink: rank rows per group
constexpr int kKB = 64;                         // shrink piece: columns of k (one 128-byte line)
constexpr int kCB = 32;                         // expand piece: output columns
constexpr int kMaxTokens = 2048;
constexpr int kMaxRank = 128;
constexpr int kPtrCache = 256;                  // (slot, slice) entries kept in shared memory
constexpr int kSTiles = 4;                      // shrink output tiles (16 x 16) per warp
constexpr int kEILP = 2;                        // expand items per warp in flight
constexpr int kSmemLimit = 227 * 1024;
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;  // bound on every wait: 200 ms

struct Args {
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    const int32_t *sorted_ids;
    const int32_t *seg;
    float *acc0, *acc1;  // [n][T][r_max] fp32 sums: buffer g & 1 this call
    int32_t *gen;        // call counter g
    int32_t *exits;      // expand CTAs that finished this call
    int32_t *err;
    int32_t T;
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int align128(int b) { return (b + 127) & ~127; }

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(saddr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(saddr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(saddr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase: false on timeout or once another warp of
// the CTA has given up.  The timer and the flag are read every 256 polls.
__device__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int32_t *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int spin = 0; spin < 256; ++spin)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitNs) return false;
    }
}

// 16 bytes global -> shared, or 16 zero bytes when !valid (src not read then).
__device__ __forceinline__ void cp16(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(saddr(dst)), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

// The mbarrier receives one arrival from this thread once all its earlier
// cp.async copies have landed (the arrival is counted in the barrier's init).
__device__ __forceinline__ void cp_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(saddr(bar)) : "memory");
}

// Small asynchronous copies for the prologue: every table load of a CTA is in
// flight at once instead of one round trip per dependent load.
__device__ __forceinline__ void cp4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(saddr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp8(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(saddr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(saddr(p)));
}

__device__ __forceinline__ uint4 lds128(const void *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ float4 lds_f4(const void *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ uint2 lds64(const void *p) { return *reinterpret_cast<const uint2 *>(p); }

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1,%2,%3,%4};" :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void stg_u2(void *p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Tables (shared memory, built by the prologue of each kernel)
// ---------------------------------------------------------------------------
struct Tables {
    int32_t *misc;    // [8]: abort flag, header words, seg[S + 1], call counter
    int32_t *seg;     // [S + 1] segment starts (sorted positions)
    int32_t *rank;    // [S] rank of a usable slot, else 0
    int32_t *tpre;    // [S] exclusive prefix of tiles per slot
    int32_t *tslot;   // [NTmax] slot of tile
    int32_t *tw;      // [NTmax + 1] exclusive prefix of tile weights
    int32_t *tok;     // [T] sorted token ids
    uint64_t *aptr;   // [S * n] when cached
    uint64_t *bptr;   // [S * n] when cached
    float *scale;     // [S] when cached
    bool cached;
};

__host__ __device__ inline bool ptrs_cached(int32_t S, int32_t n) { return S * n <= kPtrCache; }

__host__ __device__ inline size_t tables_bytes(int32_t S, int32_t n, int32_t T, int32_t TG) {
    const size_t NTmax = static_cast<size_t>(S) + (T + TG - 1) / TG;
    size_t b = 4 * (8 + (S + 1) + 2 * static_cast<size_t>(S) + NTmax + (NTmax + 1) + T);
    b = (b + 15) & ~size_t(15);
    if (ptrs_cached(S, n)) b += 16 * static_cast<size_t>(S) * n + 4 * static_cast<size_t>(S);
    return (b + 15) & ~size_t(15);
}

__device__ Tables carve_tables(unsigned char *base, int32_t S, int32_t n, int32_t T, int32_t TG) {
    const int32_t NTmax = S + (T + TG - 1) / TG;
    Tables m;
    m.misc = reinterpret_cast<int32_t *>(base);
    m.seg = m.misc + 8;
    m.rank = m.seg + S + 1;
    m.tpre = m.rank + S;
    m.tslot = m.tpre + S;
    m.tw = m.tslot + NTmax;
    m.tok = m.tw + NTmax + 1;
    size_t off = 4 * (8 + (S + 1) + 2 * static_cast<size_t>(S) + NTmax + (NTmax + 1) + T);
    off = (off + 15) & ~size_t(15);
    m.cached = ptrs_cached(S, n);
    m.aptr = reinterpret_cast<uint64_t *>(base + off);
    m.bptr = m.aptr + static_cast<size_t>(S) * n;
    m.scale = reinterpret_cast<float *>(m.bptr + static_cast<size_t>(S) * n);
    return m;
}

struct Tile {
    int32_t s, p0, len, r;
};

// Tokens per tile of a slot of rank r: kTG for the shrink; for the expand kTGe,
// halved above rank 64 so that a 16-column stage still fits its accumulator
// rows.
template <bool kExpand>
__device__ __forceinline__ int32_t tile_tokens(int32_t r) {
    return kExpand ? (r > kRG ? kTGe / 2 : kTGe) : kTG;
}

template <bool kExpand>
__device__ __forceinline__ Tile tile_at(const Tables &m, int32_t t) {
    Tile ti;
    ti.s = m.tslot[t];
    ti.r = m.rank[ti.s];
    const int32_t TG = tile_tokens<kExpand>(ti.r);
    ti.p0 = m.seg[ti.s] + (t - m.tpre[ti.s]) * TG;
    ti.len = min(TG, m.seg[ti.s + 1] - ti.p0);
    return ti;
}

// Exclusive scan of data[0..n) by one whole warp; returns the total.
__device__ int32_t warp_scan(int32_t *data, int32_t n, int lane) {
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

// Rank groups of a slot: ranks above kRG are split in two equal halves (a
// multiple of 4 rows each, as ranks are multiples of 8).
__device__ __forceinline__ int32_t rank_groups(int32_t r) { return r > kRG ? 2 : 1; }

// Pieces and weight of a piece (rows of the staged data, or their 64-byte
// equivalent) of a tile of `len` tokens and rank r.
__device__ __forceinline__ int32_t shrink_pieces(int32_t r, const Shape &sh) {
    return sh.n * rank_groups(r) * ceil_div(sh.k, kKB);
}
__device__ __forceinline__ int32_t shrink_piece_w(int32_t r, int32_t len) { return r / rank_groups(r) + len + 2; }

__device__ __forceinline__ int32_t expand_pieces(const Shape &sh) {
    int32_t c = 0;
    for (int i = 0; i < sh.n; ++i) c += ceil_div(sh.off[i + 1] - sh.off[i], kCB);
    return c;
}
__device__ __forceinline__ int32_t expand_piece_w(int32_t r, int32_t len) { return r + 2 * len + 8; }

// Prologue: all table loads as one batch of asynchronous copies, then checks,
// then warp 0 builds the tile list and its weight prefix.  The caller syncs.
template <bool kExpand>
__device__ void load_tables(const Args &a, const Shape &sh, const void *table, const Tables &m) {
    const int32_t S = sh.S, T = a.T, n = sh.n;
    const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5, lane = tid & 31;
    const TableView tab(table, S, n);
    const int32_t *hdr = static_cast<const int32_t *>(table);
    if (tid == 0) {
        cp4(m.misc + 1, hdr);
        cp4(m.misc + 2, hdr + 1);
        cp4(m.misc + 3, hdr + 2);
        cp4(m.misc + 4, a.gen);
    }
    for (int t = tid; t < T; t += nthreads) cp4(m.tok + t, a.sorted_ids + t);
    for (int s = tid; s <= S; s += nthreads) cp4(m.seg + s, a.seg + s);
    for (int s = tid; s < S; s += nthreads) cp4(m.rank + s, tab.rank + s);
    if (tid == 32) cp4(m.misc + 5, a.seg + S + 1);
    if (m.cached) {
        for (int e = tid; e < S * n; e += nthreads) {
            cp8(m.aptr + e, tab.a_ptr + e);
            cp8(m.bptr + e, tab.b_ptr + e);
        }
        if (kExpand)
            for (int s = tid; s < S; s += nthreads) cp4(m.scale + s, tab.scale + s);
    }
    cp_wait_all();
    __syncthreads();
    for (int t = tid; t < T; t += nthreads) {
        const int32_t v = m.tok[t];
        if (v < 0 || v >= T) {
            report_error(a.err, LORA_ERR_INVALID_ARG);
            m.tok[t] = -1;
        }
    }
    if (warp != 0) return;
    const bool ok = m.misc[1] == kTableMagic && m.misc[2] == S && m.misc[3] == n && m.misc[5] == T;
    if (!ok && lane == 0 && blockIdx.x == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
    for (int s = lane; s < S; s += 32) {
        const int32_t r = m.rank[s];
        const int32_t cnt = m.seg[s + 1] - m.seg[s];
        if (ok && r > sh.r_max && blockIdx.x == 0) report_error(a.err, LORA_ERR_RANK);
        const bool use = ok && cnt > 0 && r > 0 && r <= sh.r_max;
        const int32_t TG = tile_tokens<kExpand>(r);
        m.rank[s] = use ? r : 0;
        m.tpre[s] = use ? (cnt + TG - 1) / TG : 0;
    }
    __syncwarp();
    const int32_t NT = warp_scan(m.tpre, S, lane);
    const int32_t P_e = kExpand ? expand_pieces(sh) : 0;
    for (int s = lane; s < S; s += 32) {
        const int32_t r = m.rank[s];
        if (r == 0) continue;
        const int32_t TG = tile_tokens<kExpand>(r);
        const int32_t cnt = m.seg[s + 1] - m.seg[s], tiles = (cnt + TG - 1) / TG;
        for (int j = 0; j < tiles; ++j) {
            const int32_t t = m.tpre[s] + j, len = min(TG, cnt - j * TG);
            m.tslot[t] = s;
            m.tw[t] = kExpand ? P_e * expand_piece_w(r, len) : shrink_pieces(r, sh) * shrink_piece_w(r, len);
        }
    }
    __syncwarp();
    const int32_t W = warp_scan(m.tw, NT, lane);
    if (lane == 0) {
        m.tw[NT] = W;
        m.misc[6] = NT;
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Shrink
// ---------------------------------------------------------------------------
// A unit: a CTA's consecutive pieces of one (tile, slice, rank group), i.e. a
// run of `cnt` items of 64 columns of k from item kb0.  An item is staged as
// R16 + L16 lines of 128 bytes (the A rows, then the token rows of x, each
// count rounded up to the 16-row ldmatrix tiles; only the real rows are
// copied), and a stage holds kbs items.
struct SUnit {
    int32_t s, i, g, p0, len, R, kb0, cnt, R16, L16, kbs;
};

struct ShrinkWalk {
    Range rg;
    int32_t nkb;
};

// Advance to the next unit of this CTA; false when none is left.
__device__ __forceinline__ bool next_shrink_unit(ShrinkWalk &w, const Tables &m, const Shape &sh, int32_t NT,
                                                 SUnit &u) {
    auto P = [&](int32_t t) { return shrink_pieces(m.rank[m.tslot[t]], sh); };
    if (!piece_valid_var(w.rg, m.tw, NT, P)) return false;
    const Tile ti = tile_at<false>(m, w.rg.tile);
    const int32_t G = rank_groups(ti.r), kb = w.rg.idx % w.nkb, ig = w.rg.idx / w.nkb;
    u.cnt = min(pieces_left_var(w.rg, m.tw, P), w.nkb - kb);
    u.s = ti.s;
    u.i = ig / G;
    u.g = ig % G;
    u.p0 = ti.p0;
    u.len = ti.len;
    u.R = ti.r / G;
    u.kb0 = kb;
    u.R16 = (u.R + 15) & ~15;
    u.L16 = (u.len + 15) & ~15;
    u.kbs = max(1, kSSlot / ((u.R16 + u.L16) * 128));
    w.rg.idx += u.cnt;
    if (w.rg.idx >= P(w.rg.tile)) {
        ++w.rg.tile;
        w.rg.idx = 0;
    }
    return true;
}

size_t shrink_smem(int32_t S, int32_t n, int32_t T) {
    return 1024 + static_cast<size_t>(kSStages) * kSSlot + 2 * kSStages * 8 + kCWarps * 256 * 4 +
           tables_bytes(S, n, T, kTG);
}

__global__ void __maxnreg__(128) stream_shrink_kernel(Args a, Shape sh, const void *table) {
    extern __shared__ unsigned char smem_raw[];
    pdl_launch_dependents();  // the expand kernel may start its prologue on the free half of each SM
    // 1024-byte aligned ring: the XOR swizzle of the 128-byte lines is by row
    unsigned char *ring = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + kSStages * kSSlot);
    uint64_t *empty = full + kSStages;
    float *scratch = reinterpret_cast<float *>(empty + kSStages);  // [kCWarps][16 x 16]
    const Tables m = carve_tables(reinterpret_cast<unsigned char *>(scratch + kCWarps * 256), sh.S, sh.n, a.T, kTG);
    volatile int32_t *abort_flag = m.misc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TableView tab(table, sh.S, sh.n);

    load_tables<false>(a, sh, table, m);
    if (tid == 0) {
        *abort_flag = 0;
        for (int st = 0; st < kSStages; ++st) {
            mbar_init(&full[st], 32);  // one arrival per lane of the producing warp
            mbar_init(&empty[st], kCWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int32_t NT = m.misc[6];
    float *acc_buf = (m.misc[4] & 1) ? a.acc1 : a.acc0;
    ShrinkWalk walk;
    walk.nkb = ceil_div(sh.k, kKB);
    walk.rg = first_piece_var(m.tw, NT, [&](int32_t t) { return shrink_pieces(m.rank[m.tslot[t]], sh); });

    if (warp >= kCWarps) {
        // ------------------------------------------------------------ producers
        // stage it belongs to producer warp it % 4; lane = (row offset, 16-byte chunk)
        const int pw = warp - kCWarps, c = lane & 7, r0 = lane >> 3;
        int32_t it = 0;
        SUnit u;
        bool stop = false;
        while (!stop && next_shrink_unit(walk, m, sh, NT, u)) {
            const int32_t e = u.s * sh.n + u.i;
            const uint16_t *A = reinterpret_cast<const uint16_t *>(m.cached ? m.aptr[e] : tab.a_ptr[e]) +
                                static_cast<int64_t>(u.g) * u.R * sh.k;
            const int32_t rows = u.R + u.len, item_bytes = (u.R16 + u.L16) * 128;
            for (int32_t q = 0; q < u.cnt; q += u.kbs, ++it) {
                if (it % kPWarps != pw) continue;
                if (it >= kSStages &&
                    !__all_sync(0xffffffffu,
                                mbar_wait(&empty[it % kSStages], ((it / kSStages) - 1) & 1, abort_flag))) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_error(a.err, LORA_ERR_TIMEOUT);
                    }
                    stop = true;
                    break;
                }
                unsigned char *sb = ring + (it % kSStages) * kSSlot;
                const int32_t mm = min(u.kbs, u.cnt - q);
                for (int32_t ei = 0; ei < mm; ++ei) {
                    const int32_t col = (u.kb0 + q + ei) * kKB + 8 * c;
                    const bool inb = col < sh.k;
                    unsigned char *item = sb + ei * item_bytes;
#pragma unroll 4
                    for (int32_t row = r0; row < rows; row += 4) {
                        const uint16_t *src;
                        int32_t d;
                        bool v = inb;
                        if (row < u.R) {
                            src = A + static_cast<int64_t>(row) * sh.k + col;
                            d = row;
                        } else {
                            const int32_t t = m.tok[u.p0 + row - u.R];
                            v = v && t >= 0;
                            src = a.x + static_cast<int64_t>(max(t, 0)) * a.ldx + col;
                            d = u.R16 + row - u.R;
                        }
                        cp16(item + d * 128 + ((c ^ (d & 7)) << 4), v ? src : a.x, v);
                    }
                }
                cp_arrive_noinc(&full[it % kSStages]);
            }
        }
        // this warp's copies land before it exits
        cp_wait_all();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g8 = lane >> 2, q4 = lane & 3;
    float *scr = scratch + warp * 256;
    // ldmatrix lane roles: A (16 x 16): row lane & 15, chunk lane >> 4;
    // x (two n-tiles of 8 tokens): row (lane & 7) + 8 (lane >> 4), chunk (lane >> 3) & 1
    const int a_row = lane & 15, a_ch = lane >> 4;
    const int x_row = (lane & 7) + ((lane >> 4) << 3), x_ch = (lane >> 3) & 1;
    int32_t it = 0;
    SUnit u;
    bool stop = false;
    while (!stop && next_shrink_unit(walk, m, sh, NT, u)) {
        const int32_t nb = u.R16 / 16, ntp = u.L16 / 16, tiles = nb * ntp;
        // this warp's output tiles, (rank block, token block) pairs: tiles w,
        // w + 4, ... when there are more tiles than warps, else one tile and a
        // share of the k-steps
        const int32_t ksplit = tiles > kCWarps ? 1 : kCWarps / tiles;
        const int32_t kpart = tiles > kCWarps ? 0 : warp / tiles;
        int32_t rbm[kSTiles], tpm[kSTiles];
        int32_t mine = 0;
#pragma unroll
        for (int t4 = 0; t4 < kSTiles; ++t4) {
            const int32_t tile = tiles > kCWarps ? warp + t4 * kCWarps : (t4 == 0 ? warp % tiles : tiles);
            const bool v = tile < tiles && kpart < ksplit;
            rbm[t4] = v ? tile % nb : 0;
            tpm[t4] = v ? tile / nb : 0;
            if (v) mine = t4 + 1;
        }
        float acc[kSTiles][2][4];
#pragma unroll
        for (int t4 = 0; t4 < kSTiles; ++t4)
#pragma unroll
            for (int h = 0; h < 2; ++h) acc[t4][h][0] = acc[t4][h][1] = acc[t4][h][2] = acc[t4][h][3] = 0.f;
        const int32_t item_bytes = (u.R16 + u.L16) * 128;
        for (int32_t q = 0; q < u.cnt; q += u.kbs, ++it) {
            if (!mbar_wait(&full[it % kSStages], (it / kSStages) & 1, abort_flag)) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report_error(a.err, LORA_ERR_TIMEOUT);
                }
                stop = true;
                break;
            }
            const unsigned char *sb = ring + (it % kSStages) * kSSlot;
            const int32_t ksteps = min(u.kbs, u.cnt - q) * (kKB / 16);
            const int32_t k0 = (kpart * ksteps) / ksplit, k1 = ((kpart + 1) * ksteps) / ksplit;
            for (int32_t step = k0; step < k1; ++step) {
                const unsigned char *item = sb + (step >> 2) * item_bytes;
                const int32_t ch = (step & 3) * 2;  // first 16-byte chunk of this k-step
                uint32_t fa[kSTiles][4], fx[kSTiles][4];
#pragma unroll
                for (int t4 = 0; t4 < kSTiles; ++t4) {
                    if (t4 < mine) {
                        const int32_t ra = rbm[t4] * 16 + a_row, rx = u.R16 + tpm[t4] * 16 + x_row;
                        ldsm_x4(item + ra * 128 + (((ch + a_ch) ^ (ra & 7)) << 4), fa[t4][0], fa[t4][1], fa[t4][2],
                                fa[t4][3]);
                        ldsm_x4(item + rx * 128 + (((ch + x_ch) ^ (rx & 7)) << 4), fx[t4][0], fx[t4][1], fx[t4][2],
                                fx[t4][3]);
                    }
                }
#pragma unroll
                for (int t4 = 0; t4 < kSTiles; ++t4) {
                    if (t4 < mine) {
                        mma_bf16_16816(acc[t4][0], fa[t4][0], fa[t4][1], fa[t4][2], fa[t4][3], fx[t4][0], fx[t4][1]);
                        mma_bf16_16816(acc[t4][1], fa[t4][0], fa[t4][1], fa[t4][2], fa[t4][3], fx[t4][2], fx[t4][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[it % kSStages]);
        }
        if (stop) break;
        // add the unit's partial sums: transpose each 16 x 16 tile to [token][rank]
        // and add 4 ranks at a time
        float *dst_rows = acc_buf + static_cast<int64_t>(u.i) * a.T * sh.r_max + u.g * u.R;
#pragma unroll
        for (int t4 = 0; t4 < kSTiles; ++t4) {
            if (t4 >= mine) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                scr[(8 * h + 2 * q4) * 16 + g8] = acc[t4][h][0];
                scr[(8 * h + 2 * q4 + 1) * 16 + g8] = acc[t4][h][1];
                scr[(8 * h + 2 * q4) * 16 + g8 + 8] = acc[t4][h][2];
                scr[(8 * h + 2 * q4 + 1) * 16 + g8 + 8] = acc[t4][h][3];
            }
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int idx = lane + 32 * h;  // 16 tokens x 4 rank quads
                const int tl = idx >> 2, jq = idx & 3;
                const int tk = tpm[t4] * 16 + tl, row = rbm[t4] * 16 + 4 * jq;
                if (tk < u.len && row < u.R) {
                    const int32_t t = m.tok[u.p0 + tk];
                    if (t >= 0) {
                        const float4 v = *reinterpret_cast<const float4 *>(scr + tl * 16 + 4 * jq);
                        red_add_v4(dst_rows + static_cast<int64_t>(t) * sh.r_max + row, v.x, v.y, v.z, v.w);
                    }
                }
            }
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------------------------
// Expand
// ---------------------------------------------------------------------------
// A unit: a CTA's consecutive pieces of one (tile, slice), i.e. a range of
// output columns; cut into stages of ec columns.
struct EUnit {
    int32_t s, i, p0, len, r, c0, c1, ec;
};

// Stage layout of `ec` columns: B rows (ec x r bf16, pitch r*2 + 16), y rows
// (len x ec bf16, pitch ec*2 + 16), accumulator rows (len x r fp32, pitch
// r*4 + 16).
struct ELayout {
    int32_t bpitch, y_off, ypitch, acc_off, apitch, bytes;
};

__device__ __forceinline__ ELayout expand_layout(int32_t ec, int32_t r, int32_t len) {
    ELayout L;
    L.bpitch = r * 2 + 16;
    L.ypitch = ec * 2 + 16;
    L.apitch = r * 4 + 16;
    L.y_off = align128(ec * L.bpitch);
    L.acc_off = align128(L.y_off + len * L.ypitch);
    L.bytes = L.acc_off + len * L.apitch;
    return L;
}

// Widest multiple of 32 columns whose stage fits.
__device__ __forceinline__ int32_t expand_cols(int32_t r, int32_t len) {
    int32_t ec = ((kESlot - 256 - len * (r * 4 + 16) - len * 16) / (2 * r + 16 + 2 * len)) & ~31;
    ec = max(ec, 32);
    while (ec > 32 && expand_layout(ec, r, len).bytes > kESlot) ec -= 32;
    return ec;
}

struct ExpandWalk {
    Range rg;
    int32_t C;
};

__device__ __forceinline__ bool next_expand_unit(ExpandWalk &w, const Tables &m, const Shape &sh, int32_t NT,
                                                 EUnit &u) {
    if (!piece_valid(w.rg, m.tw, NT, w.C)) return false;
    const Tile ti = tile_at<true>(m, w.rg.tile);
    int32_t i = 0, cb = w.rg.idx, nb = ceil_div(sh.off[1] - sh.off[0], kCB);
    while (cb >= nb && i + 1 < sh.n) {
        cb -= nb;
        ++i;
        nb = ceil_div(sh.off[i + 1] - sh.off[i], kCB);
    }
    const int32_t cnt = min(pieces_left_in_tile(w.rg, m.tw, w.C), nb - cb);
    u.s = ti.s;
    u.i = i;
    u.p0 = ti.p0;
    u.len = ti.len;
    u.r = ti.r;
    u.c0 = cb * kCB;
    u.c1 = min((cb + cnt) * kCB, sh.off[i + 1] - sh.off[i]);
    u.ec = expand_cols(ti.r, ti.len);
    w.rg.idx += cnt;
    if (w.rg.idx >= w.C) {
        ++w.rg.tile;
        w.rg.idx = 0;
    }
    return true;
}

size_t expand_smem(int32_t S, int32_t n, int32_t T) {
    return 128 + static_cast<size_t>(kEStages) * kESlot + 2 * kEStages * 8 + tables_bytes(S, n, T, kTGe / 2);
}

__global__ void __maxnreg__(128) stream_expand_kernel(Args a, Shape sh, const void *table) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = smem_raw + ((128u - (saddr(smem_raw) & 127u)) & 127u);
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + kEStages * kESlot);
    uint64_t *empty = full + kEStages;
    const Tables m = carve_tables(reinterpret_cast<unsigned char *>(empty + kEStages), sh.S, sh.n, a.T, kTGe / 2);
    volatile int32_t *abort_flag = m.misc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TableView tab(table, sh.S, sh.n);

    load_tables<true>(a, sh, table, m);
    if (tid == 0) {
        *abort_flag = 0;
        for (int st = 0; st < kEStages; ++st) {
            mbar_init(&full[st], 32);
            mbar_init(&empty[st], kCWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int32_t NT = m.misc[6];
    const int32_t g = m.misc[4];
    const float *acc_buf = (g & 1) ? a.acc1 : a.acc0;
    // The other buffer held the previous call's sums and nothing reads it now:
    // clear this CTA's share of it for the next call.
    {
        float4 *other = reinterpret_cast<float4 *>((g & 1) ? a.acc0 : a.acc1);
        const int64_t n4 = static_cast<int64_t>(sh.n) * a.T * sh.r_max / 4;
        for (int64_t z = static_cast<int64_t>(blockIdx.x) * kThreads + tid; z < n4;
             z += static_cast<int64_t>(gridDim.x) * kThreads)
            other[z] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    ExpandWalk walk;
    walk.C = expand_pieces(sh);
    walk.rg = first_piece(m.tw, NT, walk.C);

    if (warp >= kCWarps) {
        // ------------------------------------------------------------ producers
        // B and y rows do not depend on the shrink: they are copied before the
        // wait for the shrink grid, which only the accumulator rows follow.
        const int pw = warp - kCWarps;
        int32_t it = 0;
        bool waited = false, stop = false;
        EUnit u;
        while (!stop && next_expand_unit(walk, m, sh, NT, u)) {
            const int32_t e = u.s * sh.n + u.i;
            const uint16_t *B = reinterpret_cast<const uint16_t *>(m.cached ? m.bptr[e] : tab.b_ptr[e]);
            const float *acc_rows = acc_buf + static_cast<int64_t>(u.i) * a.T * sh.r_max;
            const ELayout L = expand_layout(u.ec, u.r, u.len);
            // lane roles for rows of r/8 (B) and r/4 (accumulator) 16-byte chunks
            const int32_t cb = u.r >> 3, pb = 32 / cb, rb0 = lane / cb, chb = lane - rb0 * cb;
            const int32_t ca = u.r >> 2, pa = 32 / ca, ra0 = lane / ca, cha = lane - ra0 * ca;
            for (int32_t c0 = u.c0; c0 < u.c1; c0 += u.ec, ++it) {
                if (it % kPWarps != pw) continue;
                const int32_t EW = min(u.ec, u.c1 - c0);
                if (it >= kEStages &&
                    !__all_sync(0xffffffffu,
                                mbar_wait(&empty[it % kEStages], ((it / kEStages) - 1) & 1, abort_flag))) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_error(a.err, LORA_ERR_TIMEOUT);
                    }
                    stop = true;
                    break;
                }
                unsigned char *sb = ring + (it % kEStages) * kESlot;
                if (rb0 < pb) {
                    const uint16_t *src = B + static_cast<int64_t>(c0) * u.r + 8 * chb;
                    for (int32_t row = rb0; row < EW; row += pb)
                        cp16(sb + row * L.bpitch + 16 * chb, src + static_cast<int64_t>(row) * u.r, true);
                }
                const int32_t cy = EW >> 3;  // 16-byte chunks of a y row
                for (int32_t tt = 0; tt < u.len; ++tt) {
                    const int32_t t = m.tok[u.p0 + tt];
                    const uint16_t *src = a.y + static_cast<int64_t>(max(t, 0)) * a.ldy + sh.off[u.i] + c0;
                    for (int32_t ch = lane; ch < cy; ch += 32)
                        cp16(sb + L.y_off + tt * L.ypitch + 16 * ch, t >= 0 ? src + 8 * ch : a.y, t >= 0);
                }
                if (!waited) {
                    pdl_wait();  // the shrink grid has finished and its sums are visible
                    waited = true;
                }
                if (ra0 < pa) {
                    for (int32_t tt = ra0; tt < u.len; tt += pa) {
                        const int32_t t = m.tok[u.p0 + tt];
                        cp16(sb + L.acc_off + tt * L.apitch + 16 * cha,
                             t >= 0 ? acc_rows + static_cast<int64_t>(t) * sh.r_max + 4 * cha : acc_rows, t >= 0);
                    }
                }
                cp_arrive_noinc(&full[it % kEStages]);
            }
        }
        cp_wait_all();
    } else {
        // ------------------------------------------------------------ consumers
        // items: 16 tokens x 16 columns (a pair of MMA n-tiles); the sums enter
        // as bf16 hi + lo, the lane's B row is one output column
        const int g8 = lane >> 2, q4 = lane & 3;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        int32_t it = 0;
        EUnit u;
        bool stop = false;
        while (!stop && next_expand_unit(walk, m, sh, NT, u)) {
            const float scale = m.cached ? m.scale[u.s] : tab.scale[u.s];
            uint16_t *yrow = a.y + sh.off[u.i];
            const ELayout L = expand_layout(u.ec, u.r, u.len);
            for (int32_t c0 = u.c0; c0 < u.c1; c0 += u.ec, ++it) {
                const int32_t EW = min(u.ec, u.c1 - c0);
                if (!mbar_wait(&full[it % kEStages], (it / kEStages) & 1, abort_flag)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_error(a.err, LORA_ERR_TIMEOUT);
                    }
                    stop = true;
                    break;
                }
                const unsigned char *sB = ring + (it % kEStages) * kESlot, *sY = sB + L.y_off, *sAcc = sB + L.acc_off;
                const int32_t npairs = ceil_div(EW / 8, 2), ntt = ceil_div(u.len, 16);
                const int32_t items = ntt * npairs, kbn = ceil_div(u.r, 32);
                for (int32_t base = warp; base < items; base += kCWarps * kEILP) {
                    float acc[kEILP][2][4];
                    int32_t ttm[kEILP], pairm[kEILP];
                    bool val[kEILP];
#pragma unroll
                    for (int mm = 0; mm < kEILP; ++mm) {
                        const int32_t item = base + mm * kCWarps;
                        val[mm] = item < items;
                        ttm[mm] = item / npairs;
                        pairm[mm] = item - ttm[mm] * npairs;
#pragma unroll
                        for (int h = 0; h < 2; ++h) acc[mm][h][0] = acc[mm][h][1] = acc[mm][h][2] = acc[mm][h][3] = 0.f;
                    }
                    for (int32_t kb = 0; kb < kbn; ++kb) {
                        const int32_t j = kb * 32 + 8 * q4;
                        const bool jok = j < u.r;
                        uint4 ha[kEILP], la[kEILP], hb[kEILP], lb[kEILP], bv[kEILP][2];
#pragma unroll
                        for (int mm = 0; mm < kEILP; ++mm) {
                            const int32_t ra = ttm[mm] * 16 + g8, rb2 = ra + 8;
                            float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
                            if (val[mm] && jok && ra < u.len) {
                                a0 = lds_f4(sAcc + ra * L.apitch + j * 4);
                                a1 = lds_f4(sAcc + ra * L.apitch + j * 4 + 16);
                            }
                            if (val[mm] && jok && rb2 < u.len) {
                                b0 = lds_f4(sAcc + rb2 * L.apitch + j * 4);
                                b1 = lds_f4(sAcc + rb2 * L.apitch + j * 4 + 16);
                            }
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                // n-tile h of the pair: the lane's B row is column
                                // 16*pair + 4*(g/2) + 2h + g%2, so its outputs land on
                                // columns 16*pair + 4q + 2h + {0, 1}
                                const int32_t col = pairm[mm] * 16 + 4 * (g8 >> 1) + 2 * h + (g8 & 1);
                                bv[mm][h] = (val[mm] && jok && col < EW) ? lds128(sB + col * L.bpitch + j * 2) : z;
                            }
                            split_bf16x2(a0.x, a0.y, ha[mm].x, la[mm].x);
                            split_bf16x2(a0.z, a0.w, ha[mm].y, la[mm].y);
                            split_bf16x2(a1.x, a1.y, ha[mm].z, la[mm].z);
                            split_bf16x2(a1.z, a1.w, ha[mm].w, la[mm].w);
                            split_bf16x2(b0.x, b0.y, hb[mm].x, lb[mm].x);
                            split_bf16x2(b0.z, b0.w, hb[mm].y, lb[mm].y);
                            split_bf16x2(b1.x, b1.y, hb[mm].z, lb[mm].z);
                            split_bf16x2(b1.z, b1.w, hb[mm].w, lb[mm].w);
                        }
#pragma unroll
                        for (int mm = 0; mm < kEILP; ++mm) {
                            if (!val[mm]) continue;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                mma_bf16_16816(acc[mm][h], ha[mm].x, hb[mm].x, ha[mm].y, hb[mm].y, bv[mm][h].x,
                                               bv[mm][h].y);
                                mma_bf16_16816(acc[mm][h], la[mm].x, lb[mm].x, la[mm].y, lb[mm].y, bv[mm][h].x,
                                               bv[mm][h].y);
                            }
                        }
#pragma unroll
                        for (int mm = 0; mm < kEILP; ++mm) {
                            if (!val[mm]) continue;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                mma_bf16_16816(acc[mm][h], ha[mm].z, hb[mm].z, ha[mm].w, hb[mm].w, bv[mm][h].z,
                                               bv[mm][h].w);
                                mma_bf16_16816(acc[mm][h], la[mm].z, lb[mm].z, la[mm].w, lb[mm].w, bv[mm][h].z,
                                               bv[mm][h].w);
                            }
                        }
                    }
                    // y = y + scale * sums with one rounding; the lane owns 4 consecutive columns
#pragma unroll
                    for (int mm = 0; mm < kEILP; ++mm) {
                        if (!val[mm]) continue;
                        const int32_t col0 = pairm[mm] * 16 + 4 * q4;
                        if (col0 >= EW) continue;
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const int32_t row = ttm[mm] * 16 + g8 + 8 * half;
                            if (row >= u.len) continue;
                            const int32_t t = m.tok[u.p0 + row];
                            if (t < 0) continue;
                            const uint2 yv = lds64(sY + row * L.ypitch + col0 * 2);
                            const float v0 = fmaf(scale, acc[mm][0][2 * half + 0], bf16lo_to_f32(yv.x));
                            const float v1 = fmaf(scale, acc[mm][0][2 * half + 1], bf16hi_to_f32(yv.x));
                            const float v2 = fmaf(scale, acc[mm][1][2 * half + 0], bf16lo_to_f32(yv.y));
                            const float v3 = fmaf(scale, acc[mm][1][2 * half + 1], bf16hi_to_f32(yv.y));
                            stg_u2(yrow + static_cast<int64_t>(t) * a.ldy + c0 + col0, pack_bf16x2(v0, v1),
                                   pack_bf16x2(v2, v3));
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[it % kEStages]);
            }
        }
    }
    // the last CTA to finish advances the call counter; a CTA without work waits
    // for the shrink grid first, so the counter never moves while a shrink CTA
    // may still read it
    __syncthreads();
    if (tid == 0) {
        pdl_wait();
        __threadfence();
        if (atomicAdd(a.exits, 1) == static_cast<int32_t>(gridDim.x) - 1) {
            *a.exits = 0;
            __threadfence();
            *a.gen = g + 1;
        }
    }
}

}  // namespace

bool decode_stream_supported(int32_t T, const Shape &sh) {
    // work weights are summed in int32: bound k and d well below overflow; the
    // tables for S slots and T tokens must fit next to the ring
    return T <= kMaxTokens && sh.r_max <= kMaxRank && sh.k % 16 == 0 && sh.k <= 65536 && sh.off[sh.n] <= 65536 &&
           shrink_smem(sh.S, sh.n, T) <= static_cast<size_t>(kSmemLimit) &&
           expand_smem(sh.S, sh.n, T) <= static_cast<size_t>(kSmemLimit);
}

cudaError_t launch_decode_stream(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                 const void *table, const int32_t *sorted_ids, const int32_t *seg, float *ws,
                                 int32_t T, int32_t *err, cudaStream_t stream) {
    static int num_sms = 0;
    static bool attr_set = false;
    if (!decode_stream_supported(T, sh)) return cudaErrorNotSupported;
    if (!attr_set) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(stream_shrink_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(stream_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        // the whole unified L1 as shared memory, so that one CTA of each kernel
        // fits on an SM at once
        e = cudaFuncSetAttribute(stream_shrink_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(stream_expand_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const WorkspaceLayout L(T, sh.n, sh.r_max, sh.S);
    char *base = reinterpret_cast<char *>(ws);
    int32_t *ctrl = reinterpret_cast<int32_t *>(base);
    Args a;
    a.x = x;
    a.ldx = ldx;
    a.y = y;
    a.ldy = ldy;
    a.sorted_ids = sorted_ids;
    a.seg = seg;
    a.acc0 = reinterpret_cast<float *>(base + L.acc2_off);
    a.acc1 = reinterpret_cast<float *>(base + L.acc3_off);
    a.gen = ctrl + 2 * LORA_MAX_SLICES * static_cast<size_t>(sh.S);
    a.exits = a.gen + 1;
    a.err = err;
    a.T = T;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = shrink_smem(sh.S, sh.n, T);
    cfg.stream = stream;
    cfg.numAttrs = 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, stream_shrink_kernel, a, sh, table);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(static_cast<unsigned>(num_sms));
    cfg2.blockDim = dim3(kThreads);
    cfg2.dynamicSmemBytes = expand_smem(sh.S, sh.n, T);
    cfg2.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg2.attrs = attr;
    cfg2.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg2, stream_expand_kernel, a, sh, table);
}

}  // namespace lora
