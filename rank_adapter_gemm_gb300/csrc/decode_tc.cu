// Decode-size LoRA branch on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory): a streaming shrink kernel, then an expand
// kernel launched as its programmatic dependent.
//
// At decode the branch streams adapter weights: every active slot's A and B are
// read once while x and y are small (llama.cpp LoRA adapter page, section
// "为什么低秩增量可以「后加」": decode is bound by memory bandwidth, the cost
// being extra launches and intermediates).
//
//   * Tiles are up to 128 sorted positions of one slot.  Shrink items are
//     (tile, slice, 64-column block of k); an item stages the tile's x rows (M,
//     the tokens) and the slice's A rows (N = r_s), only real rows, the rows the
//     MMA reads past them feeding accumulator rows or columns nobody reads.
//     Items are weighted by the bytes they move and every CTA takes a
//     contiguous range of equal weight (split-K over k, TensorRT-LLM LoRA
//     serving page, "path 2: split-K tuning").  Each CTA's items of one
//     (tile, slice) form a unit whose partial sums are added into an fp32
//     accumulator in the workspace (red.global.add.v4.f32).  Four producer warps
//     gather rows with per-thread 16-byte asynchronous copies (cp.async), each
//     keeping two ring stages in flight.
//   * The expand kernel is launched as a programmatic dependent of the shrink:
//     while the shrink runs it builds its tables, clears its share of the other
//     accumulator buffer and starts copying B; it then waits for the shrink grid
//     (griddepcontrol.wait) before reading the sums.  Units are (tile, slice,
//     128 output columns), balanced by bytes, and run transposed: M = the 128
//     output columns (B rows), N = the tile's tokens, K = the rank, with the sums
//     entering as bf16 hi + lo parts (x A^T to about 2^-17 relative).  A
//     tensor-memory lane is an output column, so all four lane quarters work on
//     every unit; a thread adds its column of s * D to the tokens' y values in
//     fp32 and rounds once to bf16.
//   * The workspace holds two accumulator buffers and a call counter g: a call
//     adds into buffer g & 1 and clears buffer (g + 1) & 1, which the previous
//     call used; the expand kernel's last CTA advances g.  No CTA waits on
//     another, so no cross-CTA counter or flag is polled.
//
// Limits (the host routes other cases elsewhere): T <= 2048, r_max <= 64, and
// the tables for S slots and T tokens must fit in shared memory next to the
// stage rings.
#include <algorithm>

#include "common.cuh"
#include "schedule.cuh"
#include "tc.cuh"

namespace lora {

namespace {

constexpr int kTile = 128;                       // tokens per tile
constexpr int kKB = 64;                          // k per item: one 128-byte row
constexpr int kCW = 128;                         // output columns per expand unit (MMA M)
constexpr int kMaxTokens = 2048;
constexpr int kSmemLimit = 227 * 1024;
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;  // bound on every wait: 200 ms
constexpr int kBarBytes = 1024;                  // barriers and flags, behind a ring
constexpr int kGuard = 16 * 1024;                // readable bytes behind a ring
constexpr int kMaxRows = kTile + 64;             // staged rows of a shrink item: tokens + r_s
constexpr int kProdWarps = 4;                    // warps 1-4 in both kernels
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kEpiWarp0 = 1 + kProdWarps;        // first epilogue warp
// shrink kernel: 8 stages of 24 KB, one flush group
constexpr int kSStages = 8;
constexpr int kSSlot = 24 * 1024;
constexpr int kSThreads = 32 + kProdThreads + 128;
// expand kernel: 4 stages of 48 KB, two epilogue groups
constexpr int kEStages = 4;
constexpr int kESlot = 48 * 1024;
constexpr int kEThreads = 32 + kProdThreads + 256;
constexpr int kBarEpi = 2;                       // named barriers 2 and 3: epilogue groups

struct Args {
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    const int32_t *sorted_ids;
    const int32_t *seg;
    float *acc[2];      // [n][T][r_max] fp32 sums: buffer g & 1 this call
    int32_t *gen;       // call counter g
    int32_t *exits;     // expand CTAs that finished this call
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

// Shrink stage: KB items of one (tile, slice), each [x rows N8 | A rows r] x 128 bytes.
__device__ __forceinline__ int32_t shrink_kb_per_stage(int32_t N8, int32_t r) {
    return max(1, kSSlot / ((N8 + r) * 128));
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
// Prologue shared by both kernels
// ---------------------------------------------------------------------------
struct Smem {
    int32_t *seg, *rank, *tpre, *tslot, *tsh, *tex, *tok, *nt;
};

__device__ __forceinline__ Smem carve_tables(int32_t *base, int32_t S, int32_t T) {
    const int32_t NTmax = S + (T + kTile - 1) / kTile;
    Smem m;
    m.nt = base;                   // [8]
    m.seg = base + 8;              // [S + 1]
    m.rank = m.seg + S + 1;        // [S]
    m.tpre = m.rank + S;           // [S]
    m.tslot = m.tpre + S;          // [NTmax]
    m.tsh = m.tslot + NTmax;       // [NTmax + 1]
    m.tex = m.tsh + NTmax + 1;     // [NTmax + 1]
    m.tok = m.tex + NTmax + 1;     // [T]
    return m;
}

__host__ __device__ inline size_t table_bytes(int32_t S, int32_t T) {
    const size_t NTmax = static_cast<size_t>(S) + (T + kTile - 1) / kTile;
    return 4 * (8 + (S + 1) + 2 * S + NTmax + 2 * (NTmax + 1) + T);
}

// All threads: sorted ids and segment offsets (independent of the table header).
// Warp 0 then reads the ranks once the header shows the table holds S slots and
// builds the work tables with shuffle scans; the caller synchronises.
__device__ void load_tables(const Args &a, const Shape &sh, const void *table, Smem m, int nthreads) {
    const int32_t S = sh.S, T = a.T;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TableView tab(table, sh.S, sh.n);
    const int32_t *hdr = static_cast<const int32_t *>(table);
    const bool ok = hdr[0] == kTableMagic && hdr[1] == S && hdr[2] == sh.n && a.seg[S + 1] == T;
    for (int t = tid; t < T; t += nthreads) {
        int32_t v = a.sorted_ids[t];
        if (v < 0 || v >= T) {
            report_error(a.err, LORA_ERR_INVALID_ARG);
            v = -1;
        }
        m.tok[t] = v;
    }
    for (int s = tid; s <= S; s += nthreads) m.seg[s] = a.seg[s];
    if (warp != 0) return;
    const int32_t nkb = (sh.k + kKB - 1) / kKB;
    const int32_t C = chunks_per_tile(sh);
    if (!ok && lane == 0 && blockIdx.x == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
    for (int s = lane; s < S; s += 32) {
        const int32_t r = ok ? tab.rank[s] : 0;
        const int32_t cnt = ok ? a.seg[s + 1] - a.seg[s] : 0;
        if (r > sh.r_max && blockIdx.x == 0) report_error(a.err, LORA_ERR_RANK);
        const bool use = ok && cnt > 0 && r > 0 && r <= sh.r_max;
        m.rank[s] = use ? r : 0;
        m.tpre[s] = use ? (cnt + kTile - 1) / kTile : 0;
    }
    __syncwarp();
    const int32_t NT = warp_exclusive_scan(m.tpre, S, lane);
    for (int s = lane; s < S; s += 32) {
        const int32_t r = m.rank[s];
        if (r == 0) continue;
        const int32_t cnt = a.seg[s + 1] - a.seg[s], tiles = (cnt + kTile - 1) / kTile;
        for (int j = 0; j < tiles; ++j) {
            const int32_t t = m.tpre[s] + j, len = min(kTile, cnt - j * kTile);
            m.tslot[t] = s;
            m.tsh[t] = sh.n * nkb * (round8(len) + r);      // 128-byte rows: items x (tokens + A rows)
            m.tex[t] = C * (2 * rp_of(r) + 4 * len + 16);  // per unit: B rows, y in and out, fixed cost
        }
    }
    __syncwarp();
    const int32_t Wsh = warp_exclusive_scan(m.tsh, NT, lane);
    const int32_t Wex = warp_exclusive_scan(m.tex, NT, lane);
    if (lane == 0) {
        m.tsh[NT] = Wsh;
        m.tex[NT] = Wex;
        *m.nt = NT;
    }
    __syncwarp();
}

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Shrink kernel
// ---------------------------------------------------------------------------
// Shared memory: kSStages x kSSlot ring | barriers | row tables [4][kMaxRows] |
// misc | work tables (>= kGuard bytes behind the ring).
__global__ void __launch_bounds__(kSThreads, 1) decode_shrink_kernel(Args a, Shape sh, const void *table) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int32_t T = a.T;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kSStages * kSSlot);
    uint64_t *empty = full + kSStages;
    uint64_t *acc_full = empty + kSStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint64_t *s_rows = reinterpret_cast<uint64_t *>(smem + kSStages * kSSlot + kBarBytes);  // [4][kMaxRows]
    int32_t *misc = reinterpret_cast<int32_t *>(s_rows + kProdWarps * kMaxRows);            // [8]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
    volatile int32_t *abort_flag = misc + 1;
    const Smem m = carve_tables(misc + 8, sh.S, T);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();  // the expand kernel may start its own prologue
    const TableView tab(table, sh.S, sh.n);
    const int32_t nkb = (sh.k + kKB - 1) / kKB;
    const int32_t P_sh = sh.n * nkb;  // items per tile: slices x blocks of k
    float *acc = ((*a.gen) & 1) ? a.acc[1] : a.acc[0];

    load_tables(a, sh, table, m, kSThreads);
    if (warp == 0) {
        if (lane == 0) {
            *abort_flag = 0;
            for (int st = 0; st < kSStages; ++st) {
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
        tc::tmem_alloc(tmem_slot, 128);  // two accumulators of 64 columns
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = tc::smem_u32(smem);
    const int32_t NT = *m.nt;
    Tabs tb;
    tb.seg = m.seg;
    tb.rank = m.rank;
    tb.tslot = m.tslot;
    tb.tpre = m.tpre;
    tb.NT = NT;

    if (warp == 0) {
        // ================================================== MMA issuer: D[token, rank] += x A_i^T
        if (lane == 0) {
            int32_t it = 0, u = 0;
            bool stop = false;
            Range rg = first_piece(m.tsh, NT, P_sh);
            while (!stop && piece_valid(rg, m.tsh, NT, P_sh)) {
                const Tile ti = tile_at(tb, rg.tile);
                const int32_t kb0 = rg.idx % nkb;
                const int32_t nitems = min(pieces_left_in_tile(rg, m.tsh, P_sh), nkb - kb0);
                const int32_t N8 = round8(ti.len), kbs = shrink_kb_per_stage(N8, ti.r);
                const uint32_t idesc = tc::idesc_bf16(kTile, round16(ti.r));
                const int32_t b = u & 1;
                if (u >= 2 && !tc::mbar_wait(&acc_empty[b], ((u >> 1) - 1) & 1, abort_flag, kWaitNs)) {
                    give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                    break;
                }
                tc::fence_after_sync();
                for (int32_t q = 0; q < nitems; q += kbs, ++it) {
                    const int st = it % kSStages;
                    if (!tc::mbar_wait(&full[st], (it / kSStages) & 1, abort_flag, kWaitNs)) {
                        give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                        stop = true;
                        break;
                    }
                    tc::fence_after_sync();
                    const int32_t mm = min(kbs, nitems - q);
                    for (int32_t e = 0; e < mm; ++e) {
                        const uint32_t xs = sbase + st * kSSlot + e * (N8 + ti.r) * 128;
                        const uint32_t as = xs + N8 * 128;
#pragma unroll
                        for (int kk = 0; kk < kKB / 16; ++kk)
                            tc::mma_bf16(tmem + b * 64, tc::smem_desc(xs + 32 * kk, 1024, tc::kLayoutSW128),
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
            tc::mma_commit(drain);
            if (!tc::mbar_wait_timed(drain, 0, kWaitNs)) report_error(a.err, LORA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        // ================================================== producers
        // Warp pw takes stages it with it % 4 == pw and publishes each one once
        // its next stage is issued (cp.async.wait_group 1), so two of its stages
        // are in flight; the last one is published after the loop.
        const int pw = warp - 1;
        int32_t it = 0, pending = -1;
        bool stop = false;
        auto publish = [&](int32_t st_it) {
            tc::fence_async_smem();
            tc::mbar_arrive(&full[st_it % kSStages]);
        };
        Range rg = first_piece(m.tsh, NT, P_sh);
        while (!stop && piece_valid(rg, m.tsh, NT, P_sh)) {
            const Tile ti = tile_at(tb, rg.tile);
            const int32_t kb0 = rg.idx % nkb, slice = rg.idx / nkb;
            const int32_t nitems = min(pieces_left_in_tile(rg, m.tsh, P_sh), nkb - kb0);
            const int32_t N8 = round8(ti.len), kbs = shrink_kb_per_stage(N8, ti.r);
            const int c = lane & 7, r0 = lane >> 3;  // this lane's 16-byte column and first row
            const int32_t rows = ti.len + ti.r;
            // this warp's row table for the unit: address of each staged row's
            // element 0 (0 = a token out of range: the row reads as zero); token
            // rows first, then the slice's A rows
            uint64_t *tbl = s_rows + pw * kMaxRows;
            __syncwarp();
            const uint64_t abase = tab.a_ptr[ti.s * sh.n + slice];
            for (int32_t row = lane; row < rows; row += 32) {
                uint64_t src;
                if (row < ti.len) {
                    const int32_t t = m.tok[ti.p0 + row];
                    src = t >= 0 ? reinterpret_cast<uint64_t>(a.x + static_cast<int64_t>(t) * a.ldx) : 0;
                } else {
                    src = abase + static_cast<uint64_t>(row - ti.len) * sh.k * 2;
                }
                tbl[row] = src;
            }
            __syncwarp();
            for (int32_t q = 0; q < nitems; q += kbs, ++it) {
                if (it % kProdWarps != pw) continue;
                if (it >= kSStages &&
                    !__all_sync(0xffffffffu, tc::mbar_wait(&empty[it % kSStages], ((it / kSStages) - 1) & 1,
                                                           abort_flag, kWaitNs))) {
                    give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                    stop = true;
                    break;
                }
                const uint32_t sb = sbase + (it % kSStages) * kSSlot;
                const int32_t mm = min(kbs, nitems - q);
                for (int32_t e = 0; e < mm; ++e) {
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
                tc::cp_commit();
                if (pending >= 0) {
                    tc::cp_wait_group<1>();
                    publish(pending);
                }
                pending = it;
            }
            rg.idx += nitems;
            if (rg.idx >= P_sh) {
                ++rg.tile;
                rg.idx = 0;
            }
        }
        tc::cp_wait_all();
        if (pending >= 0) publish(pending);
    } else {
        // ================================================== flush: partial sums -> acc (lane = token)
        const int q = warp & 3, gt = 32 * q + lane;
        int32_t u = 0;
        bool stop = false;
        Range rg = first_piece(m.tsh, NT, P_sh);
        while (!stop && piece_valid(rg, m.tsh, NT, P_sh)) {
            const Tile ti = tile_at(tb, rg.tile);
            const int32_t kb0 = rg.idx % nkb, slice = rg.idx / nkb;
            const int32_t nitems = min(pieces_left_in_tile(rg, m.tsh, P_sh), nkb - kb0);
            const int32_t b = u & 1, this_u = u++;
            rg.idx += nitems;
            if (rg.idx >= P_sh) {
                ++rg.tile;
                rg.idx = 0;
            }
            const bool fail =
                !__all_sync(0xffffffffu, tc::mbar_wait(&acc_full[b], (this_u >> 1) & 1, abort_flag, kWaitNs));
            if (fail) give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
            tc::fence_after_sync();
            if (!fail && 32 * q < ti.len) {
                const int32_t t = gt < ti.len ? m.tok[ti.p0 + gt] : -1;
                uint32_t v[64];
                const int32_t R16 = round16(ti.r);
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    if (16 * h < R16)
                        tc::tmem_ld16_async(tmem + (static_cast<uint32_t>(32 * q) << 16) + b * 64 + 16 * h, v + 16 * h);
                tc::tmem_wait_ld64(v);
                if (t >= 0) {
                    float *dst = acc + (static_cast<int64_t>(slice) * T + t) * sh.r_max;
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (4 * e < ti.r)
                            red_add_v4(dst + 4 * e, __uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                       __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                }
            }
            tc::fence_before_sync();
            stop = named_sync_or(kBarEpi, 128, fail || *abort_flag);
            if (gt == 0) tc::mbar_arrive(&acc_empty[b]);
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 128);
    }
}

// ---------------------------------------------------------------------------
// Expand kernel (programmatic dependent of the shrink)
// ---------------------------------------------------------------------------
// Shared memory: kEStages x kESlot ring | barriers | misc | work tables.
__global__ void __launch_bounds__(kEThreads, 1) decode_expand_kernel(Args a, Shape sh, const void *table) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int32_t T = a.T;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kEStages * kESlot);
    uint64_t *empty = full + kEStages;
    uint64_t *acc_full = empty + kEStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    int32_t *misc = reinterpret_cast<int32_t *>(smem + kEStages * kESlot + kBarBytes);  // [8]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
    volatile int32_t *abort_flag = misc + 1;
    const Smem m = carve_tables(misc + 8, sh.S, T);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TableView tab(table, sh.S, sh.n);
    const int32_t C = chunks_per_tile(sh);
    const int32_t g = *a.gen;
    const float *acc = (g & 1) ? a.acc[1] : a.acc[0];

    load_tables(a, sh, table, m, kEThreads);
    // The other buffer held the previous call's sums and nothing reads it now:
    // clear this CTA's share of it for the next call.
    {
        float4 *other = reinterpret_cast<float4 *>((g & 1) ? a.acc[0] : a.acc[1]);
        const int64_t n4 = static_cast<int64_t>(sh.n) * T * sh.r_max / 4;
        for (int64_t z = static_cast<int64_t>(blockIdx.x) * kEThreads + tid; z < n4;
             z += static_cast<int64_t>(gridDim.x) * kEThreads)
            other[z] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (warp == 0) {
        if (lane == 0) {
            *abort_flag = 0;
            for (int st = 0; st < kEStages; ++st) {
                tc::mbar_init(&full[st], 32);
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
        tc::tmem_alloc(tmem_slot, 256);  // two accumulators of 128 columns
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = tc::smem_u32(smem);
    const int32_t NT = *m.nt;
    Tabs tb;
    tb.seg = m.seg;
    tb.rank = m.rank;
    tb.tslot = m.tslot;
    tb.tpre = m.tpre;
    tb.NT = NT;

    if (warp == 0) {
        // ================================================== MMA issuer: D[column, token] = B xa_hi^T + B xa_lo^T
        if (lane == 0) {
            int32_t it = 0;
            Range re = first_piece(m.tex, NT, C);
            while (piece_valid(re, m.tex, NT, C)) {
                const Tile ti = tile_at(tb, re.tile);
                const uint32_t rowb = rowb_of(ti.r);
                const uint32_t layout = tc::layout_for_rowb(rowb);
                const int32_t N16 = round16(ti.len);
                const uint32_t bsz = kCW * rowb, xsz = round1k(static_cast<uint32_t>(N16) * rowb);
                const uint32_t idesc = tc::idesc_bf16(kCW, N16);
                const int32_t b = it & 1;
                const int st = it % kEStages;
                if ((it >= 2 && !tc::mbar_wait(&acc_empty[b], ((it >> 1) - 1) & 1, abort_flag, kWaitNs)) ||
                    !tc::mbar_wait(&full[st], (it / kEStages) & 1, abort_flag, kWaitNs)) {
                    give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t ob = sbase + st * kESlot;
                const int32_t ksteps = rp_of(ti.r) / 16;
                for (int kk = 0; kk < ksteps; ++kk) {
                    // K steps of 16 within a swizzled row: +32 bytes
                    const uint64_t ad = tc::smem_desc(ob + 32 * kk, 8 * rowb, layout);
                    tc::mma_bf16(tmem + b * 128, ad, tc::smem_desc(ob + bsz + 32 * kk, 8 * rowb, layout), idesc, kk > 0);
                    tc::mma_bf16(tmem + b * 128, ad, tc::smem_desc(ob + bsz + xsz + 32 * kk, 8 * rowb, layout), idesc,
                                 true);
                }
                tc::mma_commit(&empty[st]);
                tc::mma_commit(&acc_full[b]);
                ++it;
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
        // Stage it (one unit) belongs to warp it % 4.  B rows are copied before
        // the shrink grid is waited for (they do not depend on it); the sums are
        // read after, split into bf16 hi and lo and stored into the stage.
        const int pw = warp - 1;
        int32_t it = 0;
        bool waited = false, stop = false;
        Range re = first_piece(m.tex, NT, C);
        while (!stop && piece_valid(re, m.tex, NT, C)) {
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
            if (this_it >= kEStages &&
                !__all_sync(0xffffffffu, tc::mbar_wait(&empty[this_it % kEStages], ((this_it / kEStages) - 1) & 1,
                                                       abort_flag, kWaitNs))) {
                give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
                stop = true;
                break;
            }
            const uint32_t ob = sbase + (this_it % kEStages) * kESlot;
            // B rows (output columns) of the chunk; ranks j >= r_s read as zero
            const uint16_t *B = reinterpret_cast<const uint16_t *>(tab.b_ptr[ti.s * sh.n + i]);
            for (int32_t z = lane; z < (width << cpr_log); z += 32) {
                const int32_t mrow = z >> cpr_log, cc = z & ((1 << cpr_log) - 1);
                const bool v = 8 * cc < ti.r;
                tc::cp16(ob + tc::swz_offset(mrow, cc, rowb), v ? B + static_cast<int64_t>(c0 + mrow) * ti.r + 8 * cc : a.x,
                         v);
            }
            tc::cp_commit();
            if (!waited) {
                pdl_wait();  // the shrink grid is complete and its sums are visible
                waited = true;
            }
            // the tile's sums of slice i as bf16 hi and lo (zero for ranks >= r_s),
            // eight independent loads in flight per lane
            const float *accr = acc + static_cast<int64_t>(i) * T * sh.r_max;
            const int32_t ngrp = ti.len * 16;
            for (int32_t z0 = 0; z0 < ngrp; z0 += 32 * 8) {
                float4 v[8];
#pragma unroll
                for (int u8 = 0; u8 < 8; ++u8) {
                    const int32_t z = z0 + lane + 32 * u8, row = z >> 4, j = 4 * (z & 15);
                    v[u8] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (z < ngrp && j < ti.r) {
                        const int32_t t = m.tok[ti.p0 + row];
                        if (t >= 0) v[u8] = ldg_cg_f4(accr + static_cast<int64_t>(t) * sh.r_max + j);
                    }
                }
#pragma unroll
                for (int u8 = 0; u8 < 8; ++u8) {
                    const int32_t z = z0 + lane + 32 * u8, row = z >> 4, j = 4 * (z & 15);
                    if (z < ngrp && j < rp) {
                        uint32_t h0, l0, h1, l1;
                        split_bf16x2(v[u8].x, v[u8].y, h0, l0);
                        split_bf16x2(v[u8].z, v[u8].w, h1, l1);
                        const uint32_t d = tc::swz_offset(row, j >> 3, rowb) + (j & 7) * 2;
                        asm volatile("st.shared.v2.u32 [%0], {%1,%2};" :: "r"(ob + bsz + d), "r"(h0), "r"(h1) : "memory");
                        asm volatile("st.shared.v2.u32 [%0], {%1,%2};" :: "r"(ob + bsz + xsz + d), "r"(l0), "r"(l1)
                                     : "memory");
                    }
                }
            }
            tc::cp_wait_all();
            tc::fence_async_smem();
            tc::mbar_arrive(&full[this_it % kEStages]);
        }
        tc::cp_wait_all();
    } else {
        // ================================================== epilogue
        // Two groups of four warps take alternate units (and accumulators); warp q
        // of a group reads tensor-memory lanes 32q..32q+31 = output columns.
        const int ew = warp - kEpiWarp0, q = warp & 3, grp = ew >> 2;
        const int bar_id = kBarEpi + grp;
        const int gt = 32 * q + lane;
        int32_t u = 0;
        bool stop = false;
        Range re = first_piece(m.tex, NT, C);
        while (!stop && piece_valid(re, m.tex, NT, C)) {
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
            // in flight while the current ones are added and stored (y is not
            // written by the shrink, so it may be read before the sums are ready)
            auto load_y = [&](int32_t t0, uint32_t (&dst)[32]) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int32_t tt = t0 + e;
                    const int32_t t = tt < ti.len ? m.tok[ti.p0 + tt] : -1;
                    dst[e] = (colv && t >= 0) ? ldg_u16(ycol + static_cast<int64_t>(t) * a.ldy) : 0u;
                }
            };
            uint32_t yv[32];
            load_y(0, yv);
            const bool fail =
                !__all_sync(0xffffffffu, tc::mbar_wait(&acc_full[b], (this_u >> 1) & 1, abort_flag, kWaitNs));
            if (fail) give_up(a.err, abort_flag, LORA_ERR_TIMEOUT);
            tc::fence_after_sync();
            if (!fail) {
                const int32_t N16 = round16(ti.len);
                for (int32_t t0 = 0; t0 < ti.len; t0 += 32) {
                    uint32_t v[32];
                    tc::tmem_ld16_async(tmem + (static_cast<uint32_t>(32 * q) << 16) + b * 128 + t0, v);
                    if (t0 + 16 < N16)
                        tc::tmem_ld16_async(tmem + (static_cast<uint32_t>(32 * q) << 16) + b * 128 + t0 + 16, v + 16);
                    tc::tmem_wait_ld32(v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = add_scaled1(yv[e], __uint_as_float(v[e]), sc);
                    if (t0 + 32 < ti.len) load_y(t0 + 32, yv);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int32_t tt = t0 + e;
                        const int32_t t = tt < ti.len ? m.tok[ti.p0 + tt] : -1;
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
        tc::tmem_dealloc(tmem, 256);
    }
    // the last CTA to finish advances the call counter for the next call; a CTA
    // without work waits for the shrink grid first, so the counter never moves
    // while a shrink CTA may still read it
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

size_t shrink_smem(int32_t S, int32_t T) {
    const size_t behind = kBarBytes + 8 * kProdWarps * kMaxRows + 32 + table_bytes(S, T);
    return 1024 + static_cast<size_t>(kSStages) * kSSlot + std::max<size_t>(behind, kGuard);
}

size_t expand_smem(int32_t S, int32_t T) {
    const size_t behind = kBarBytes + 32 + table_bytes(S, T);
    return 1024 + static_cast<size_t>(kEStages) * kESlot + std::max<size_t>(behind, kGuard);
}

}  // namespace

bool decode_tc_supported(int32_t T, const Shape &sh) {
    // the work weights are summed in int32: bound d and k well below overflow;
    // the tables for S slots and T tokens must fit next to the stage rings
    return T <= kMaxTokens && sh.r_max <= 64 && sh.off[sh.n] <= 65536 && sh.k <= 65536 &&
           shrink_smem(sh.S, T) <= static_cast<size_t>(kSmemLimit) &&
           expand_smem(sh.S, T) <= static_cast<size_t>(kSmemLimit);
}

cudaError_t launch_decode_tc(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                             const void *table, const int32_t *sorted_ids, const int32_t *seg, float *ws, int32_t T,
                             int32_t *err, cudaStream_t stream) {
    static int num_sms = 0;
    static bool attr_set = false;
    if (!decode_tc_supported(T, sh)) return cudaErrorNotSupported;
    if (!attr_set) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(decode_shrink_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(decode_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
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
    a.acc[0] = reinterpret_cast<float *>(base + L.acc2_off);
    a.acc[1] = reinterpret_cast<float *>(base + L.acc3_off);
    a.gen = ctrl + 2 * LORA_MAX_SLICES * static_cast<size_t>(sh.S);
    a.exits = a.gen + 1;
    a.err = err;
    a.T = T;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms));
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = shrink_smem(sh.S, T);
    cfg.stream = stream;
    cfg.numAttrs = 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_shrink_kernel, a, sh, table);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(static_cast<unsigned>(num_sms));
    cfg2.blockDim = dim3(kEThreads);
    cfg2.dynamicSmemBytes = expand_smem(sh.S, T);
    cfg2.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg2.attrs = attr;
    cfg2.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg2, decode_expand_kernel, a, sh, table);
}

}  // namespace lora
