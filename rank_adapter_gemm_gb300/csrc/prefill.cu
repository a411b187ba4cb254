// Prefill-size LoRA branch on the 5th-generation tensor cores (tcgen05, with
// the accumulators in tensor memory).
//
// Long segments (many tokens of one slot, as in a prompt) make both halves of
// the branch real dense contractions: the shrink xa = x A^T has M = tokens,
// N = rank, K = k, and the expand y += s (xa) B^T has M = tokens, N = output
// columns, K = rank (TensorRT-LLM LoRA serving page, "path 3: eager mode":
// prefill batches take the grouped-GEMM operator, not the decode graph path).
// Both stay bound by HBM (x for the shrink, the y read-modify-write for the
// expand), but the multiply-add rate they need at that bandwidth is above what
// the CUDA cores give, so the products run on the tensor cores.
//
// Tiles are 128 consecutive sorted positions of one slot's segment (the MMA M),
// so every tile multiplies by a single adapter.  Token rows are gathered through
// sorted_ids with per-thread asynchronous 16-byte copies (cp.async) straight into
// the swizzled shared-memory layout the tensor cores read; a tile never needs its
// rows to be contiguous in x or y.
//
// Shrink: one cluster of KS CTAs per tile splits k (split-K, TensorRT-LLM LoRA
// serving page, "path 2: split-K tuning": M small against K gives too few
// blocks).  Each CTA runs a 4- to 8-stage copy pipeline feeding one MMA thread, the
// partial [128 x n*RP] sums meet through distributed shared memory in rank order
// (deterministic), and xa is written as two bf16 parts, hi + lo (xa to about
// 2^-17 relative), in sorted order: [n][T][RP].
//
// Expand: a persistent CTA per SM walks units (tile, slice, 256 output columns).
// One warp stages the unit's xa hi/lo and B tiles, one thread issues
// D = xa_hi B^T + xa_lo B^T into one of two tensor-memory accumulators, two
// warps stream the unit's y rows into a ring of 16 KB buffers, and eight warps
// (two groups taking alternate buffers) read the accumulator (one token row per
// thread), add it to y in fp32, round once to bf16 and write the rows back with
// coalesced stores.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "tc.cuh"

namespace lora {

namespace {

constexpr int kTile = 128;                      // tokens per tile (MMA M)
constexpr int kKB = 64;                         // k per shrink stage: one 128-byte row
constexpr int kXStage = kTile * kKB * 2;        // 16 KB of x per stage
constexpr int kCols = 256;                      // output columns per expand unit (MMA N)
constexpr int kSub = 64;                        // output columns per y buffer
constexpr int kYBuf = kTile * kSub * 2;         // 16 KB
constexpr uint64_t kWaitNs = 2000000000ull;     // bound on every wait: 2 s
constexpr int kShrinkThreads = 160;             // warps 0-3 copy + epilogue, warp 4 MMA
constexpr int kEpiWarps = 8;                    // expand epilogue: two groups of four warps
constexpr int kExpandThreads = 128 + 32 * kEpiWarps;  // warp 0 MMA, 1 operands, 2-3 y, 4-11 epilogue
constexpr int kSmemLimit = 227 * 1024;
constexpr int kClaimRing = 8;                   // expand: ring of the CTA's claimed unit ids

struct PrefillArgs {
    // x as [T][k] in boxes of 128 rows x 64 columns (128-byte swizzle): the
    // shrink's x tile when the tile's 128 sorted positions are consecutive rows
    CUtensorMap xmap;
    // slice i of y as [T][d_i]: loads of 128 rows x 64 columns and stores of 32
    // rows x 64 columns (128-byte swizzle), for units whose rows are consecutive
    CUtensorMap yload[LORA_MAX_SLICES];
    CUtensorMap ystore[LORA_MAX_SLICES];
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    const int32_t *sorted_ids;
    const int32_t *seg;
    uint16_t *xa_hi;  // [n][T][RP]
    uint16_t *xa_lo;
    int32_t *claim;   // the expand's unit counter (a workspace word the shrink sets to 0)
    int32_t T;
    int32_t *err;
};

__device__ __forceinline__ int32_t tiles_of(int32_t cnt, int32_t) { return (cnt + kTile - 1) / kTile; }

// Tile `tile` of the prefix table: slot, first sorted position and length.
struct TileInfo {
    int32_t s, p0, len;
};

__device__ __forceinline__ TileInfo tile_info(const int32_t *s_pref, const int32_t *seg, int32_t S, int32_t tile) {
    TileInfo ti;
    ti.s = find_slot(s_pref, S, tile);
    const int32_t start = seg[ti.s], end = seg[ti.s + 1];
    ti.p0 = start + (tile - s_pref[ti.s]) * kTile;
    ti.len = min(kTile, end - ti.p0);
    return ti;
}

// Records a timeout once and tells the other roles to stop.
__device__ __forceinline__ void give_up(int32_t *err, volatile int32_t *abort_flag) {
    report_error(err, LORA_ERR_TIMEOUT);
    *abort_flag = 1;
}

__device__ __forceinline__ uint4 lds_u4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_u4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void sts_f4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Tensor-map store of a 2-D box from shared memory, in this thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const void *map, int32_t x, int32_t y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(map), "r"(x), "r"(y), "r"(src) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// y (8 bf16 in v) + s * acc[0..8) in fp32, rounded once to bf16.
__device__ __forceinline__ uint4 add_scaled(uint4 v, const uint32_t *acc, float s) {
    uint4 o;
    o.x = pack_bf16x2(bf16lo_to_f32(v.x) + s * __uint_as_float(acc[0]), bf16hi_to_f32(v.x) + s * __uint_as_float(acc[1]));
    o.y = pack_bf16x2(bf16lo_to_f32(v.y) + s * __uint_as_float(acc[2]), bf16hi_to_f32(v.y) + s * __uint_as_float(acc[3]));
    o.z = pack_bf16x2(bf16lo_to_f32(v.z) + s * __uint_as_float(acc[4]), bf16hi_to_f32(v.z) + s * __uint_as_float(acc[5]));
    o.w = pack_bf16x2(bf16lo_to_f32(v.w) + s * __uint_as_float(acc[6]), bf16hi_to_f32(v.w) + s * __uint_as_float(acc[7]));
    return o;
}

// Tensor-memory columns to allocate: a power of two >= 32.
__host__ __device__ constexpr uint32_t tmem_cols_for(int c) {
    return c <= 32 ? 32u : (c <= 64 ? 64u : (c <= 128 ? 128u : (c <= 256 ? 256u : 512u)));
}

// ---------------------------------------------------------------------------
// Shrink
// ---------------------------------------------------------------------------
// Shared memory (base rounded up to 1024 bytes): `stages` x [x 128x64 | A_i RPx64
// for each slice], all 128-byte swizzled K-major; then barriers and tables.  After
// the main loop the stage area holds the fp32 partial [128][n*RP + 4].
template <int RP>
__global__ void __launch_bounds__(kShrinkThreads) tc_shrink_kernel(const __grid_constant__ PrefillArgs a, Shape sh,
                                                                   const void *table, int32_t stages) {
    // the expand of this call claims its units from a counter that starts at 0
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *a.claim = 0;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int n = sh.n, NC = n * RP;
    const uint32_t stage_bytes = kXStage + NC * kKB * 2;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + stages * stage_bytes);
    uint64_t *empty = full + stages;
    uint64_t *done = empty + stages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int32_t *abort_flag = reinterpret_cast<int32_t *>(tmem_slot + 1);
    int32_t *s_tok = reinterpret_cast<int32_t *>(tmem_slot + 2);  // [kTile]
    int32_t *s_pref = s_tok + kTile;                               // [S]
    int32_t *s_scr = s_pref + sh.S;                                // [33]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TableView tab(table, sh.S, sh.n);
    const int32_t total = slot_item_prefix(table, sh, a.seg, a.T, s_pref, s_scr, a.err, tiles_of);
    const int32_t tile = blockIdx.y;
    if (tile >= total) return;  // the same for every CTA of the cluster

    const TileInfo ti = tile_info(s_pref, a.seg, sh.S, tile);
    const int32_t r_s = tab.rank[ti.s];
    const uint32_t KS = cluster_nctarank(), crank = cluster_ctarank();
    const int32_t nkb = (sh.k + kKB - 1) / kKB;
    const int32_t kb_lo = static_cast<int32_t>(crank * nkb / KS);
    const int32_t nloc = static_cast<int32_t>((crank + 1) * nkb / KS) - kb_lo;
    const uint32_t tcols = tmem_cols_for(NC);

    // A tile whose sorted positions hold consecutive rows of x (the tokens of
    // one request in a prefill batch) takes its x rows as one tensor-map copy
    // per k-block; other tiles gather them row by row.
    const int32_t first = a.sorted_ids[ti.p0];
    bool row_ok = true;
    if (threadIdx.x < kTile) {
        int32_t t = -1;
        if (static_cast<int32_t>(threadIdx.x) < ti.len) {
            t = a.sorted_ids[ti.p0 + threadIdx.x];
            if (t < 0 || t >= a.T) {
                report_error(a.err, LORA_ERR_INVALID_ARG);
                t = -1;
            }
            row_ok = t >= 0 && t == first + static_cast<int32_t>(threadIdx.x);
        }
        s_tok[threadIdx.x] = t;
    }
    if (warp == 4) {
        if (lane == 0) {
            for (int st = 0; st < stages; ++st) {
                tc::mbar_init(&full[st], kTile);
                tc::mbar_init(&empty[st], 1);
            }
            tc::mbar_init(done, 1);
            *abort_flag = 0;
            tc::mbar_init_fence();
        }
        __syncwarp();
        tc::tmem_alloc(tmem_slot, tcols);
        tc::fence_before_sync();
    }
    const bool contig = __syncthreads_and(row_ok) != 0;
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = tc::smem_u32(smem);

    if (warp < 4) {
        // ---- producers: x rows (gathered) and the A rows of every slice ----
        const int tid = threadIdx.x;
        // A stage is published (this thread's copies of it landed) before the
        // thread waits for the slot it refills next, so the MMA of stage s
        // waits for the MMA of stage s - 2 (or earlier), not s - 1
        const int depth = stages - 1;
        int32_t issued = 0, published = 0;
        for (int32_t it = 0; it < nloc; ++it) {
            if (it >= depth) {
                tc::cp_wait_group_n(depth - 1);
                tc::fence_async_smem();
                tc::mbar_arrive(&full[(it - depth) % stages]);
                published = it - depth + 1;
            }
            const int st = it % stages;
            if (it >= stages && !tc::mbar_wait(&empty[st], ((it / stages) - 1) & 1, abort_flag, kWaitNs)) {
                give_up(a.err, abort_flag);
                break;
            }
            const int32_t c0 = (kb_lo + it) * kKB;
            const uint32_t xs = sbase + st * stage_bytes;
            if (contig) {
                // rows past the tile are other tokens' x or the map's zero fill:
                // their sums are never read
                if (tid == 0) {
                    tc::mbar_expect_tx(&full[st], kXStage);
                    tc::tma_load_2d(xs, &a.xmap, c0, first, &full[st]);
                }
            } else {
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int q = tid + kTile * m, row = q >> 3, c = q & 7;
                    const int32_t t = s_tok[row], col = c0 + 8 * c;
                    const bool v = t >= 0 && col < sh.k;
                    tc::cp16(xs + tc::swz_offset(row, c, 128), v ? a.x + static_cast<int64_t>(t) * a.ldx + col : a.x,
                             v);
                }
            }
            for (int q = tid; q < NC * 8; q += kTile) {
                const int i = q / (RP * 8), j = (q >> 3) % RP, c = q & 7;
                const int32_t col = c0 + 8 * c;
                const bool v = j < r_s && col < sh.k;
                const uint16_t *A = reinterpret_cast<const uint16_t *>(tab.a_ptr[ti.s * n + i]);
                tc::cp16(xs + kXStage + i * RP * 128 + tc::swz_offset(j, c, 128),
                     v ? A + static_cast<int64_t>(j) * sh.k + col : a.x, v);
            }
            tc::cp_commit();
            issued = it + 1;
        }
        tc::cp_wait_all();
        tc::fence_async_smem();
        for (int32_t it = published; it < issued; ++it) tc::mbar_arrive(&full[it % stages]);
    } else {
        // ---- MMA issuer: D[:, i*RP .. +RP) += x_tile A_i^T over this CTA's k range;
        // the slices' A rows sit back to back in the stage, so one MMA of N = n RP
        // covers them all ----
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kTile, NC);
            for (int32_t it = 0; it < nloc; ++it) {
                const int st = it % stages;
                if (!tc::mbar_wait(&full[st], (it / stages) & 1, abort_flag, kWaitNs)) {
                    give_up(a.err, abort_flag);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t xs = sbase + st * stage_bytes;
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk)
                    tc::mma_bf16(tmem, tc::smem_desc(xs + 32 * kk, 1024, tc::kLayoutSW128),
                                 tc::smem_desc(xs + kXStage + 32 * kk, 1024, tc::kLayoutSW128), idesc, it > 0 || kk > 0);
                tc::mma_commit(&empty[st]);
            }
            tc::mma_commit(done);  // arrives once every MMA issued above has completed
        }
        __syncwarp();  // the whole warp reaches the cluster barrier together
    }

    // ---- epilogue: tensor memory -> fp32 partial rows in shared memory ----
    const int pitch = NC + 4;  // floats; the 16-byte skew spreads rows over banks
    const uint32_t part = sbase;
    if (warp < 4) {
        const bool ok = __all_sync(0xffffffffu, tc::mbar_wait_timed(done, 0, kWaitNs));
        if (!ok) give_up(a.err, abort_flag);
        tc::fence_after_sync();
        const int row = warp * 32 + lane;
        for (int cb = 0; cb < NC; cb += 16) {
            uint32_t r[16];
            tc::tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cb, r);
            const bool use = ok && nloc > 0 && !*abort_flag;
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                sts_f4(part + 4u * (row * pitch + cb + e), use ? __uint_as_float(r[e]) : 0.f,
                       use ? __uint_as_float(r[e + 1]) : 0.f, use ? __uint_as_float(r[e + 2]) : 0.f,
                       use ? __uint_as_float(r[e + 3]) : 0.f);
        }
        tc::fence_before_sync();
    }
    cluster_sync();

    // ---- split-K reduction in rank order, then xa as bf16 hi + lo ----
    {
        const int r_lo = static_cast<int>(crank * kTile / KS);
        const int r_hi = min(ti.len, static_cast<int>((crank + 1) * kTile / KS));
        const int groups = NC / 4;
        for (int e = threadIdx.x; e < (r_hi - r_lo) * groups; e += blockDim.x) {
            const int row = r_lo + e / groups, col = 4 * (e % groups);
            const uint32_t off = part + 4u * (row * pitch + col);
            float4 acc = ld_dsmem_f4(map_to_rank(off, 0));
            for (uint32_t c = 1; c < KS; ++c) {
                const float4 v = ld_dsmem_f4(map_to_rank(off, c));
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            uint32_t h0, l0, h1, l1;
            split_bf16x2(acc.x, acc.y, h0, l0);
            split_bf16x2(acc.z, acc.w, h1, l1);
            const int i = col / RP, j = col % RP;
            const size_t o = (static_cast<size_t>(i) * a.T + ti.p0 + row) * RP + j;
            *reinterpret_cast<uint2 *>(a.xa_hi + o) = make_uint2(h0, h1);
            *reinterpret_cast<uint2 *>(a.xa_lo + o) = make_uint2(l0, l1);
        }
    }
    cluster_sync();  // no CTA leaves while another still reads its partial
    if (warp == 4) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, tcols);
    }
}

// ---------------------------------------------------------------------------
// Expand
// ---------------------------------------------------------------------------
struct Unit {
    int32_t s, i, p0, len, c0, width;
};

// Chunks of kCols output columns: prefix per slice.
struct ChunkPrefix {
    int32_t pre[LORA_MAX_SLICES + 1];
};

__device__ __forceinline__ Unit unit_info(int64_t u, int32_t per_tile, const ChunkPrefix &cp, const Shape &sh,
                                          const int32_t *s_pref, const int32_t *seg) {
    const int32_t tile = static_cast<int32_t>(u / per_tile), w = static_cast<int32_t>(u % per_tile);
    const TileInfo ti = tile_info(s_pref, seg, sh.S, tile);
    int i = 0;
    while (i + 1 < sh.n && cp.pre[i + 1] <= w) ++i;
    Unit un;
    un.s = ti.s;
    un.i = i;
    un.p0 = ti.p0;
    un.len = ti.len;
    un.c0 = (w - cp.pre[i]) * kCols;
    un.width = min(kCols, sh.off[i + 1] - sh.off[i] - un.c0);
    return un;
}

// Shared memory (base rounded up to 1024 bytes): two operand stages of
// [xa_hi 128xRP | xa_lo 128xRP | B 256xRP] (rows of RP*2 bytes, swizzled to that
// width), `ystages` (even) y buffers of 128 rows x 128 bytes (128-byte swizzle),
// then barriers, the tile table and the segment offsets.
template <int RP>
__global__ void __launch_bounds__(kExpandThreads, 1) tc_expand_kernel(const __grid_constant__ PrefillArgs a, Shape sh,
                                                                      const void *table, int32_t ystages) {
    constexpr int rowb = RP * 2;
    constexpr uint32_t layout = rowb == 128 ? tc::kLayoutSW128 : (rowb == 64 ? tc::kLayoutSW64 : tc::kLayoutSW32);
    constexpr int xa_bytes = kTile * rowb;
    constexpr int op_bytes = 2 * xa_bytes + kCols * rowb;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *op_full = reinterpret_cast<uint64_t *>(smem + 2 * op_bytes + ystages * kYBuf);
    uint64_t *op_empty = op_full + 2;
    uint64_t *acc_full = op_empty + 2;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint64_t *y_full = drain + 1;
    uint64_t *y_empty = y_full + ystages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(y_empty + ystages);
    volatile int32_t *abort_flag = reinterpret_cast<int32_t *>(tmem_slot + 1);
    int32_t *s_pref = reinterpret_cast<int32_t *>(tmem_slot + 2);  // [S]
    int32_t *s_scr = s_pref + sh.S;                                // [40]
    int32_t *s_seg = s_scr + 40;                                   // [S + 1]
    volatile int32_t *s_q = s_seg + sh.S + 1;                      // [kClaimRing] claimed unit ids
    volatile int32_t *s_nq = s_q + kClaimRing;                     // ring entries published

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const TableView tab(table, sh.S, sh.n);
    const int32_t ntiles = slot_item_prefix(table, sh, a.seg, a.T, s_pref, s_scr, a.err, tiles_of);
    for (int i = threadIdx.x; i <= sh.S; i += blockDim.x) s_seg[i] = a.seg[i];
    ChunkPrefix cp;
    cp.pre[0] = 0;
    for (int i = 0; i < LORA_MAX_SLICES; ++i)
        cp.pre[i + 1] = cp.pre[i] + (i < sh.n ? (sh.off[i + 1] - sh.off[i] + kCols - 1) / kCols : 0);
    const int32_t per_tile = cp.pre[sh.n];
    const int64_t U = static_cast<int64_t>(ntiles) * per_tile;
    if (U >= (int64_t(1) << 30)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
        return;
    }
    // Units are claimed, not split up front: CTA b starts with unit b and then takes
    // the next unclaimed one (gridDim.x + the counter), so an SM that streams faster
    // does more of them.  The operand warp claims; entry j of the ring holds the
    // CTA's j-th unit (-1 once none is left).  Every reader is at most four units
    // behind the operand warp (its ring of operand stages, the MMA's two
    // accumulators, the epilogue's release of them), so an entry is reused only
    // after everyone has read it.
    if (static_cast<int64_t>(blockIdx.x) >= U) return;
    auto claimed = [&](int32_t j) -> int32_t {
        if (*s_nq <= j) {
            const uint64_t t0 = globaltimer_ns();
            while (*s_nq <= j) {
                if (*abort_flag) return -1;
                if (globaltimer_ns() - t0 > kWaitNs) {
                    give_up(a.err, abort_flag);
                    return -1;
                }
                __nanosleep(32);
            }
        }
        __threadfence_block();
        return s_q[j % kClaimRing];
    };

    if (warp == 0) {
        if (lane == 0) {
            for (int b = 0; b < 2; ++b) {
                tc::mbar_init(&op_full[b], 32);
                tc::mbar_init(&op_empty[b], 1);
                tc::mbar_init(&acc_full[b], 1);
                tc::mbar_init(&acc_empty[b], kEpiWarps);
            }
            tc::mbar_init(drain, 1);
            for (int b = 0; b < ystages; ++b) {
                tc::mbar_init(&y_full[b], 64);
                tc::mbar_init(&y_empty[b], 4);
            }
            *abort_flag = 0;
            s_q[0] = static_cast<int32_t>(blockIdx.x);
            *s_nq = 1;
            tc::mbar_init_fence();
        }
        __syncwarp();
        tc::tmem_alloc(tmem_slot, 2 * kCols);
        tc::fence_before_sync();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = tc::smem_u32(smem);
    const uint32_t ybase = sbase + 2 * op_bytes;

    if (warp == 0) {
        // ---- MMA issuer: acc[b] = xa_hi B^T + xa_lo B^T ----
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kTile, kCols);
            for (int32_t it = 0; claimed(it) >= 0; ++it) {
                const int32_t b = it & 1;
                if (!tc::mbar_wait(&op_full[b], (it >> 1) & 1, abort_flag, kWaitNs) ||
                    (it >= 2 && !tc::mbar_wait(&acc_empty[b], ((it >> 1) - 1) & 1, abort_flag, kWaitNs))) {
                    give_up(a.err, abort_flag);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t ob = sbase + b * op_bytes;
#pragma unroll
                for (int kk = 0; kk < RP / 16; ++kk) {
                    const uint64_t bd = tc::smem_desc(ob + 2 * xa_bytes + 32 * kk, 8 * rowb, layout);
                    tc::mma_bf16(tmem + b * kCols, tc::smem_desc(ob + 32 * kk, 8 * rowb, layout), bd, idesc, kk > 0);
                    tc::mma_bf16(tmem + b * kCols, tc::smem_desc(ob + xa_bytes + 32 * kk, 8 * rowb, layout), bd, idesc,
                                 true);
                }
                tc::mma_commit(&op_empty[b]);
                tc::mma_commit(&acc_full[b]);
            }
            tc::mma_commit(drain);
            if (!tc::mbar_wait_timed(drain, 0, kWaitNs)) report_error(a.err, LORA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- operands: xa hi/lo rows of the tile and the B rows of the chunk;
        // lane 0 claims the next unit while this one's copies are in flight ----
        int32_t u = static_cast<int32_t>(blockIdx.x);
        for (int32_t it = 0; u >= 0; ++it) {
            const int32_t b = it & 1;
            const Unit un = unit_info(u, per_tile, cp, sh, s_pref, s_seg);
            int32_t nxt = -1;
            if (lane == 0) {
                const int64_t v = static_cast<int64_t>(atomicAdd(a.claim, 1)) + gridDim.x;
                nxt = v < U ? static_cast<int32_t>(v) : -1;
            }
            const int32_t r_s = tab.rank[un.s];
            const uint16_t *B = reinterpret_cast<const uint16_t *>(tab.b_ptr[un.s * sh.n + un.i]);
            if (it >= 2 && !tc::mbar_wait(&op_empty[b], ((it >> 1) - 1) & 1, abort_flag, kWaitNs)) {
                give_up(a.err, abort_flag);
                break;
            }
            const uint32_t ob = sbase + b * op_bytes;
            constexpr int cpr = rowb / 16;  // 16-byte chunks per row
            const size_t xrow = static_cast<size_t>(un.i) * a.T + un.p0;
            for (int q = lane; q < kTile * cpr; q += 32) {
                const int row = q / cpr, c = q % cpr;
                const bool v = row < un.len;
                const size_t o = (xrow + row) * RP + 8 * c;
                const uint32_t d = tc::swz_offset(row, c, rowb);
                tc::cp16(ob + d, v ? a.xa_hi + o : a.xa_hi, v);
                tc::cp16(ob + xa_bytes + d, v ? a.xa_lo + o : a.xa_lo, v);
            }
            for (int q = lane; q < kCols * cpr; q += 32) {
                const int m = q / cpr, c = q % cpr;
                const bool v = m < un.width && 8 * c < r_s;
                tc::cp16(ob + 2 * xa_bytes + tc::swz_offset(m, c, rowb),
                         v ? B + static_cast<int64_t>(un.c0 + m) * r_s + 8 * c : a.xa_hi, v);
            }
            tc::cp_wait_all();
            tc::fence_async_smem();
            if (lane == 0) {
                s_q[(it + 1) % kClaimRing] = nxt;
                __threadfence_block();
                *s_nq = it + 2;
            }
            tc::mbar_arrive(&op_full[b]);
            u = __shfl_sync(0xffffffffu, nxt, 0);
        }
        tc::cp_wait_all();
    } else if (warp < 4) {
        // ---- y rows of the unit, 64 columns per buffer; the next unit's token
        // ids are fetched while this unit's copies are issued ----
        // A unit whose rows are consecutive rows of y takes each buffer as one
        // tensor-map copy (thread 0); otherwise 16-byte copies per row.
        const int yt = threadIdx.x - 64;  // 0..63
        int32_t yit = 0;
        bool stop = false;
        int32_t tok[16], tok_next[16];
        int2 ends = make_int2(0, 0), ends_next = make_int2(0, 0);  // the unit's first and last token ids
        int32_t u_next = claimed(0);
        Unit un_next = unit_info(u_next >= 0 ? u_next : 0, per_tile, cp, sh, s_pref, s_seg);
        auto fetch = [&](const Unit &un, int32_t (&dst)[16]) {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int row = (yt >> 3) + 8 * m;
                const int32_t t = row < un.len ? a.sorted_ids[un.p0 + row] : -1;
                dst[m] = t < a.T ? t : -1;
            }
            return make_int2(a.sorted_ids[un.p0], a.sorted_ids[un.p0 + un.len - 1]);
        };
        if (u_next >= 0) ends_next = fetch(un_next, tok_next);
        for (int32_t it = 0; u_next >= 0 && !stop; ++it) {
            const Unit un = un_next;
            ends = ends_next;
#pragma unroll
            for (int m = 0; m < 16; ++m) tok[m] = tok_next[m];
            // a slot's sorted positions hold strictly increasing token ids (the sort
            // is stable), so first and last ids len - 1 apart mean consecutive rows
            const int32_t first = ends.x;
            const bool contig = ends.x >= 0 && ends.y < a.T && ends.y - ends.x == un.len - 1;
            const int nsub = (un.width + kSub - 1) / kSub;
            for (int q = 0; q < nsub; ++q, ++yit) {
                const int yb = yit % ystages;
                if (yit >= ystages && !tc::mbar_wait(&y_empty[yb], ((yit / ystages) - 1) & 1, abort_flag, kWaitNs)) {
                    give_up(a.err, abort_flag);
                    stop = true;
                    break;
                }
                const uint32_t dst = ybase + yb * kYBuf;
                if (contig) {
                    // rows past the unit are other tokens' y or the map's zero fill: never stored
                    if (yt == 0) {
                        tc::mbar_expect_tx(&y_full[yb], kYBuf);
                        tc::tma_load_2d(dst, &a.yload[un.i], un.c0 + q * kSub, first, &y_full[yb]);
                    }
                } else {
                    const int c = yt & 7, col = q * kSub + 8 * c;
                    const uint16_t *ycol = a.y + sh.off[un.i] + un.c0 + col;
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const int row = (yt >> 3) + 8 * m;
                        if (tok[m] >= 0 && col < un.width)
                            tc::cp16(dst + tc::swz_offset(row, c, 128), ycol + static_cast<int64_t>(tok[m]) * a.ldy,
                                     true);
                    }
                }
                tc::cp_arrive_noinc(&y_full[yb]);
            }
            // the next unit once this one's copies are issued
            u_next = stop ? -1 : claimed(it + 1);
            if (u_next >= 0) {
                un_next = unit_info(u_next, per_tile, cp, sh, s_pref, s_seg);
                ends_next = fetch(un_next, tok_next);
            }
        }
        tc::cp_wait_all();
    } else {
        // ---- epilogue: two groups of four warps take alternate y buffers; in
        // each group a warp owns 32 token rows (its tensor-memory lane quarter)
        // and a thread one row ----
        const int eq = warp & 3, grp = (warp - 4) >> 2, row = 32 * eq + lane;
        int32_t yit = 0;
        bool stop = false;
        int32_t u_next = claimed(0);
        Unit un_next = unit_info(u_next >= 0 ? u_next : 0, per_tile, cp, sh, s_pref, s_seg);
        int32_t t_next = u_next >= 0 && row < un_next.len ? a.sorted_ids[un_next.p0 + row] : -1;
        for (int32_t it = 0; u_next >= 0 && !stop; ++it) {
            const int32_t b = it & 1;
            const Unit un = un_next;
            const int32_t t = t_next < a.T ? t_next : -1;
            u_next = claimed(it + 1);
            if (u_next >= 0) {
                un_next = unit_info(u_next, per_tile, cp, sh, s_pref, s_seg);
                t_next = row < un_next.len ? a.sorted_ids[un_next.p0 + row] : -1;
            }
            if (!__all_sync(0xffffffffu, tc::mbar_wait(&acc_full[b], (it >> 1) & 1, abort_flag, kWaitNs))) {
                give_up(a.err, abort_flag);
                break;
            }
            tc::fence_after_sync();
            const float sc = tab.scale[un.s];
            // this warp's 32 rows consecutive rows of y: one tensor-map store per buffer
            const int32_t first_w = __shfl_sync(0xffffffffu, t, 0);
            const bool wcontig = __all_sync(0xffffffffu, t >= 0 && t == first_w + lane);
            const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * eq) << 16) + b * kCols;
            uint16_t *yrow = a.y + sh.off[un.i] + un.c0;
            const int nsub = (un.width + kSub - 1) / kSub;
            for (int q = 0; q < nsub; ++q, ++yit) {
                if ((yit & 1) != grp) continue;
                const int yb = yit % ystages;
                if (!__all_sync(0xffffffffu, tc::mbar_wait(&y_full[yb], (yit / ystages) & 1, abort_flag, kWaitNs))) {
                    give_up(a.err, abort_flag);
                    stop = true;
                    break;
                }
                const uint32_t ys = ybase + yb * kYBuf;
                uint32_t acc[64];
#pragma unroll
                for (int h = 0; h < kSub / 16; ++h) tc::tmem_ld16_async(tbase + q * kSub + 16 * h, acc + 16 * h);
                tc::tmem_wait_ld64(acc);
                if (t >= 0) {
#pragma unroll
                    for (int c = 0; c < kSub / 8; ++c) {
                        if (q * kSub + 8 * c < un.width) {
                            const uint32_t addr = ys + tc::swz_offset(row, c, 128);
                            sts_u4(addr, add_scaled(lds_u4(addr), acc + 8 * c, sc));
                        }
                    }
                }
                if (wcontig) {
                    // columns past the slice are clipped by the slice's map
                    tc::fence_async_smem();  // the rows (generic proxy) before the store reads them
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&a.ystore[un.i], un.c0 + q * kSub, first_w, ys + 32 * eq * 128);
                        bulk_commit();
                        bulk_wait_read();  // the buffer may be refilled once the store has read it
                    }
                    __syncwarp();
                } else {
                    __syncwarp();
                    // coalesced write-back of this warp's 32 rows: 4 rows x 128 bytes per step
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const int rr = (lane >> 3) + 4 * m, c = lane & 7;
                        const int32_t tr = __shfl_sync(0xffffffffu, t, rr);
                        const int col = q * kSub + 8 * c;
                        if (tr >= 0 && col < un.width) {
                            const uint4 v = lds_u4(ys + tc::swz_offset(32 * eq + rr, c, 128));
                            stg_u4(yrow + static_cast<int64_t>(tr) * a.ldy + col, v);
                        }
                    }
                    __syncwarp();
                }
                if (lane == 0) tc::mbar_arrive(&y_empty[yb]);
            }
            if (stop) break;
            tc::fence_before_sync();
            if (lane == 0) tc::mbar_arrive(&acc_empty[b]);
        }
        if (lane == 0) bulk_wait_all();  // the stores are complete before the CTA leaves
    }
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 2 * kCols);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
size_t table_words(int32_t S) { return sizeof(int32_t) * (2 * static_cast<size_t>(S) + 48 + kClaimRing + 8); }

size_t shrink_smem(int RP, int n, int stages, int32_t S) {
    return 1024 + static_cast<size_t>(stages) * (kXStage + n * RP * kKB * 2) + 8 * (2 * stages + 1) + 8 +
           sizeof(int32_t) * kTile + table_words(S);
}

// About 100 KB of stages (two CTAs per SM where they fit), at least 4.
int shrink_stages(int RP, int n, int32_t S) {
    const int stage = kXStage + n * RP * kKB * 2;
    int st = std::min(8, std::max(4, (100 * 1024) / stage));
    for (; st >= 3; --st)
        if (shrink_smem(RP, n, st, S) <= static_cast<size_t>(kSmemLimit)) return st;
    return 0;
}

size_t expand_smem(int RP, int ystages, int32_t S) {
    return 1024 + 2 * static_cast<size_t>(1024 * RP) + static_cast<size_t>(ystages) * kYBuf +
           8 * (9 + 2 * ystages) + 8 + table_words(S);
}

// An even number of y buffers (the two epilogue groups take alternate ones).
int expand_ystages(int RP, int32_t S) {
    for (int ys = 8; ys >= 2; ys -= 2)
        if (expand_smem(RP, ys, S) <= static_cast<size_t>(kSmemLimit)) return ys;
    return 0;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int RP>
cudaError_t launch_rp(const PrefillArgs &a, const Shape &sh, const void *table, cudaStream_t stream) {
    // per call: the attributes belong to the current device's context
    cudaError_t e = cudaFuncSetAttribute(tc_shrink_kernel<RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc_expand_kernel<RP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;

    // shrink: (KS, tiles) with clusters of KS CTAs along k
    const int stages = shrink_stages(RP, sh.n, sh.S);
    const int ys = expand_ystages(RP, sh.S);
    if (stages == 0 || ys == 0) return cudaErrorInvalidConfiguration;
    const int64_t tiles_bound = ceil_div(a.T, kTile) + std::min<int64_t>(sh.S, a.T);
    const int64_t tiles_est = ceil_div(a.T, kTile);
    const int64_t nkb = ceil_div(sh.k, kKB);
    int64_t ks = (4 * sms) / std::max<int64_t>(1, tiles_est);
    ks = std::max<int64_t>(1, std::min<int64_t>({ks, 8, std::max<int64_t>(1, nkb / 2)}));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ks), static_cast<unsigned>(tiles_bound));
    cfg.blockDim = dim3(kShrinkThreads);
    cfg.dynamicSmemBytes = shrink_smem(RP, sh.n, stages, sh.S);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ks);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, tc_shrink_kernel<RP>, a, sh, table, int32_t(stages));
    if (e != cudaSuccess) return e;

    // expand: one persistent CTA per SM
    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(static_cast<unsigned>(sms));
    cfg2.blockDim = dim3(kExpandThreads);
    cfg2.dynamicSmemBytes = expand_smem(RP, ys, sh.S);
    cfg2.stream = stream;
    cfg2.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg2, tc_expand_kernel<RP>, a, sh, table, int32_t(ys));
}

}  // namespace

bool encode_bf16_rows_map(CUtensorMap *m, const void *base, int64_t ld, int32_t rows, int32_t cols, int32_t box_rows,
                          int32_t box_cols, bool swizzle128);

bool prefill_supported(int32_t r_max) { return r_max <= 64; }

cudaError_t launch_prefill(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                           const void *table, const int32_t *sorted_ids, const int32_t *seg, float *ws, int32_t T,
                           int32_t *err, cudaStream_t stream) {
    if (!prefill_supported(sh.r_max)) return cudaErrorNotSupported;
    const WorkspaceLayout L(T, sh.n, sh.r_max, sh.S);
    char *w = reinterpret_cast<char *>(ws);
    PrefillArgs a;
    std::memset(&a, 0, sizeof a);
    // (a map needs at least one row; with T = 0 no tile reads it)
    if (!encode_bf16_rows_map(&a.xmap, x, ldx, std::max(T, 1), sh.k, kTile, kKB, true)) return cudaErrorNotSupported;
    for (int i = 0; i < sh.n; ++i) {
        const int32_t di = sh.off[i + 1] - sh.off[i];
        if (!encode_bf16_rows_map(&a.yload[i], y + sh.off[i], ldy, std::max(T, 1), di, kTile, kSub, true) ||
            !encode_bf16_rows_map(&a.ystore[i], y + sh.off[i], ldy, std::max(T, 1), di, 32, kSub, true))
            return cudaErrorNotSupported;
    }
    a.x = x;
    a.ldx = ldx;
    a.y = y;
    a.ldy = ldy;
    a.sorted_ids = sorted_ids;
    a.seg = seg;
    a.xa_hi = reinterpret_cast<uint16_t *>(w + L.hi_off);
    a.xa_lo = reinterpret_cast<uint16_t *>(w + L.lo_off);
    // a global word of the workspace's control area that no other path of a
    // prefill call uses
    a.claim = reinterpret_cast<int32_t *>(w) + 2 * LORA_MAX_SLICES * static_cast<size_t>(sh.S) + 8;
    a.T = T;
    a.err = err;
    switch (tc_rank_pad(sh.r_max)) {
    case 16: return launch_rp<16>(a, sh, table, stream);
    case 32: return launch_rp<32>(a, sh, table, stream);
    default: return launch_rp<64>(a, sh, table, stream);
    }
}

}  // namespace lora
