// Decode-size LoRA branch as one persistent kernel per call that streams the
// adapter tiles with TMA (LORA_PATH_DECODE_TMA).
//
// At decode the branch reads every active adapter's A and B once while x and y
// are small (llama.cpp LoRA adapter page, section "为什么低秩增量可以「后加」":
// the low-rank branch is bandwidth-bound at decode).  A call therefore has to
// keep HBM busy from its first microsecond to its last, and the fixed costs of
// a call (launch, first burst, the shrink -> expand dependency, the tail) are
// what separates it from the roofline.  The kernel is built around that:
//
//   * Two CTAs per SM, about 110 KB of shared memory each: one CTA's loads
//     stay in flight while the other waits on its tensor cores or writes y.
//     The call is launched as a programmatic dependent, so a CTA of the next
//     call takes an SM slot as soon as one of this call's CTAs there exits;
//     its producer warp issues the first stages of adapter weights before
//     griddepcontrol.wait (the weights never depend on the previous layer),
//     so their first burst overlaps the previous call's tail.  Only x, y and
//     the workspace wait for the previous grid.
//   * Stages of up to 32 KB in a ring of three, one mbarrier each.  A shrink
//     stage holds, for one slot, one group of its tokens and a run of 64-wide
//     k-blocks: the group's x rows (16-byte cp.async copies, gathered through
//     sorted_ids by a second warp into the 128-byte swizzled layout), then
//     every slice's A rows (TMA 2D boxes of [r][64] bf16, 128-byte swizzle, one
//     per slice and k-block).  An expand stage holds up to `eu` units of one
//     slice: [128 columns][rp ranks] boxes of B (rp = the rank rounded up to 16,
//     32 or 64, with the matching swizzle; ranks past r are the tensor map's
//     zero fill), then the group's y rows of those columns.
//   * The 5th-generation tensor cores do the arithmetic (tcgen05.mma, bf16
//     operands straight from the swizzled stage tiles, fp32 accumulators in
//     tensor memory), issued by one thread: a shrink run (one slot, one token
//     group, consecutive k-blocks) accumulates D[128 tokens][n r ranks] over
//     its stages, each stage released by tcgen05.commit once its MMAs have read
//     it; at the end of the run four warps read D and add it into an fp32
//     buffer (red.global.add.v4) - the split over k follows the byte-balanced
//     partition (TensorRT-LLM LoRA serving page, "路径二:split-K 调优").  A
//     per-slot counter of finished k-blocks (release / acquire) tells the
//     expand of that slot, in the same kernel, that its sums are complete; the
//     expand's B tiles are already streaming meanwhile.
//   * An expand unit is 128 output columns of one slice: D[128 columns][tokens]
//     = B box x sums^T, the sums rounded once to bf16 (2^-9 relative, what
//     serving engines' expand kernels take) in a swizzled tile, two tensor-
//     memory buffers so that the next unit's MMAs overlap this unit's
//     epilogue, which writes y = bf16(y + s * acc), rounded once.
//   * The work of a call is described by a plan built once per batch and
//     slot table (lora_build_plan(s)): the active slots with their token
//     groups, and for every CTA its contiguous share of the shrink pieces
//     (slot, token group, k-block) and of the expand units (slot, token group,
//     slice, 64 output columns), each list split by the bytes it moves.
//   * The workspace holds two sum buffers and two sets of counters selected by
//     a call counter g: call g adds into set g & 1 and clears set (g + 1) & 1,
//     which call g - 1 used; the last CTA to finish advances g.
//
// Every wait is bounded (globaltimer).  A slot whose sums do not complete
// within 200 ms is reported as LORA_ERR_TIMEOUT and its y rows are left as
// they were; the ring keeps running so the CTA drains and exits normally.
#include <algorithm>
#include <cstring>

#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace lora {

// ---------------------------------------------------------------------------
// Slot table with tensor maps: the ordinary table (TableLayout), then a
// 128-byte block header {magic, S, n, k, slice offsets}, per-slot flags, and
// for every slot eight CUtensorMaps of 128 bytes.  A is read as k-blocks of
// 64 columns: a map over rows x k viewed as [k / 64][rows][64] (box of `depth`
// k-blocks x rows x 64, 128-byte swizzle), which lands in shared memory as
// `depth` consecutive [rows][64] tiles.  When the slot's slices are one
// packed [n r][k] block (flag kSlotPackedA), maps 0..3 cover all n r rows with
// depths 1, 2, 4 and 8, so a stage of k-blocks takes one to four copies;
// otherwise map i covers slice i with depth 1.  Maps 4 + i: B_s,i as [d_i][r]
// (box [128][rp], rp = r rounded up to 16, 32 or 64 with the 32-, 64- or
// 128-byte swizzle, ranks past r zero-filled).
// ---------------------------------------------------------------------------
constexpr int32_t kTmaTableMagic = 0x4d414d54;

constexpr int32_t kSlotPackedA = 1;
constexpr int kMapsPerSlot = 8;

struct TmaTableLayout {
    size_t hdr, flags, maps, bytes;
    __host__ __device__ TmaTableLayout(int32_t S, int32_t n) {
        (void)n;
        hdr = (TableLayout(S, n).bytes + 127) & ~size_t(127);
        flags = hdr + 128;
        maps = flags + ((size_t(S) * 4 + 127) & ~size_t(127));
        bytes = maps + size_t(S) * kMapsPerSlot * 128;
    }
};

namespace {

constexpr int kThreads = 192;        // warp 0: TMA, warp 1: row gather, warps 2..5: tensor cores
constexpr int kMmaThreads = 128;
constexpr int kStages = 3;
constexpr int kStageBytes = 32768;   // 256 rows of 128 bytes
constexpr int kXaBytes = 64 * 64 * 2;  // expand sums of up to 64 tokens x 64 ranks, bf16
constexpr int kSmemBytes = kStages * kStageBytes + kXaBytes + 1024;  // + alignment slack
constexpr int kTmemCols = 256;       // shrink D (ranks 0..127 at column 0, 128.. at 128), then the expand's
                                     // two 64-column buffers
                                     // (two CTAs of 256 columns share an SM's 512)
constexpr int kUnitCols = 128;       // expand unit: output columns
constexpr int kMaxGrid = 512;
constexpr int kCtasPerSm = 2;      // two CTAs of a call share an SM (about 110 KB of shared memory each)
constexpr int kMaxRank = 64;
constexpr int kMaxNR = 192;          // n_slices * r_max
constexpr int kGe = 64;              // expand token group
constexpr int32_t kPlanMagic = 0x4e4c5054;
constexpr uint64_t kRingLimitNs = 1000ull * 1000 * 1000;
constexpr uint64_t kSlotLimitNs = 200ull * 1000 * 1000;

// Plan layout: header | slot records [S] | CTA records [kMaxGrid] | sorted ids [T].
struct PlanHdr {
    int32_t magic, T, S, n, k, r_max, na, grid;
    int32_t off[LORA_MAX_SLICES + 1];
    int32_t nkb, ublk, pad0, pad1;
    uint64_t table;
    int32_t pad[12];
};
static_assert(sizeof(PlanHdr) == 128, "plan header");

struct SlotRec {
    int32_t s, seg0, cnt, r;
    float scale;
    int32_t gs, ngs, cs;   // shrink: token group size, groups, k-blocks per stage
    int32_t ge, nge;       // expand: token group size, groups
    int32_t wps, wpe;      // weight of one shrink piece / expand unit (16-byte units)
    int32_t rp, eu;        // B box width in ranks (16, 32 or 64), expand units per stage
    int32_t pk, pad;       // A slices packed (one copy per stage covers every slice)
};
static_assert(sizeof(SlotRec) == 64, "slot record");

struct CtaRec {
    int32_t s_tile, s_idx, s_count, pad0;
    int32_t e_tile, e_idx, e_count, pad1;
};
static_assert(sizeof(CtaRec) == 32, "CTA record");

__host__ __device__ inline size_t plan_slots_off() { return sizeof(PlanHdr); }
__host__ __device__ inline size_t plan_ctas_off(int32_t S) { return plan_slots_off() + size_t(S) * sizeof(SlotRec); }
__host__ __device__ inline size_t plan_ids_off(int32_t S) { return plan_ctas_off(S) + size_t(kMaxGrid) * sizeof(CtaRec); }
__host__ __device__ inline size_t plan_total(int32_t T, int32_t S) { return tma_plan_size(T, S); }
static_assert(sizeof(PlanHdr) + sizeof(CtaRec) * kMaxGrid == 128 + 512 * 32, "plan layout matches tma_plan_size");

__host__ __device__ inline int32_t cdiv(int32_t a, int32_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int32_t pad16i(int32_t v) { return (v + 15) & ~15; }
// Rows of an expand unit's y tile in the stage: the group rounded up to 8.
__host__ __device__ inline int32_t ytile_rows(int32_t gsz) { return (gsz + 7) & ~7; }
constexpr int32_t kGatherCost = 88;  // a four-row gather's fixed cost beyond its 512 bytes (16-byte units)
constexpr int32_t kUnitCost = 1536;  // an expand unit's fixed cost (16-byte units)
constexpr int32_t kShrinkStageCost = 1600;  // a shrink stage's fixed cost, shared by its k-blocks (16-byte units)
// Width in ranks of a slot's B boxes (the rank rounded up to 16, 32 or 64;
// ranks past r are the tensor map's zero fill).
__host__ __device__ inline int32_t b_box_ranks(int32_t r) { return r <= 16 ? 16 : (r <= 32 ? 32 : 64); }

struct TArgs {
    // x as [T][k] (box [1][64], 128-byte swizzle) for the four-row gathers
    CUtensorMap xmap;
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    const unsigned char *plan;
    float *acc0, *acc1;        // [T][n r_max] fp32 sums (token-major), set g & 1 this call
    int32_t *done0, *done1;    // [S] finished k-blocks per slot
    int32_t *gen, *exits;      // call counter, CTAs that finished this call
    int32_t *err;
    int32_t T, S, n, k, r_max;
    int32_t xdiv;              // x row of y row p: p / xdiv (routed experts sharing a token's x)
    int32_t off[LORA_MAX_SLICES + 1];
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sa(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait on a phase of a ring barrier; false after kRingLimitNs or once
// another role has given up (*abort set), which only a broken device causes.
// The MMA warps poll without pause (they have nothing else to do and the
// stage's data is what they wait for); the copy warps, whose waits end when an
// MMA warp frees a slot, sleep `backoff_ns` between polls so that their
// spinning takes no issue slots from the MMA warps of their sub-partitions.
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, volatile int32_t *abort,
                                          uint32_t backoff_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 16; ++i) {
            if (mbar_try_wait(bar, parity)) return true;
            if (backoff_ns) __nanosleep(backoff_ns);
        }
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kRingLimitNs) {
            *abort = 1;
            return false;
        }
    }
}
constexpr uint32_t kCopyBackoffNs = 128;


// 16 bytes global -> shared through L2, or 16 zero bytes when !valid.
__device__ __forceinline__ void cp16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
// Arrive on `bar` once this thread's earlier cp.async copies have landed (the
// barrier's count includes the arrival).
__device__ __forceinline__ void cp_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void stg128(void *p, uint4 v) {
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;"
        :: "r"(dst), "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, int32_t x, int32_t y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy) : "memory");
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void mma_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Barrier of the four tensor-core warps that also ORs a predicate over them:
// every decision that changes their control flow goes through it, so that
// they always meet at the same barriers.
__device__ __forceinline__ bool mma_any(bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(p ? 1u : 0u) : "memory");
    return r != 0;
}
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Four rows (token ids rows.x .. rows.w) of a box one row high, stored as
// four consecutive rows of the box width at dst.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void *map, int32_t col, int4 rows, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        :: "r"(dst), "l"(map), "r"(col), "r"(rows.x), "r"(rows.y), "r"(rows.z), "r"(rows.w), "r"(bar) : "memory");
}
// Token ids of rows 4 q .. 4 q + 3 of a group of gsz rows whose ids are in
// shared memory; rows past the group repeat its last id (those tile rows are
// never used).
__device__ __forceinline__ int4 four_ids(const int32_t *ids, int32_t q, int32_t gsz) {
    const int32_t r = 4 * q;
    return make_int4(ids[min(r, gsz - 1)], ids[min(r + 1, gsz - 1)], ids[min(r + 2, gsz - 1)],
                     ids[min(r + 3, gsz - 1)]);
}



// ---------------------------------------------------------------------------
// Walking a CTA's share of the plan
// ---------------------------------------------------------------------------
struct Slot {
    int32_t s, seg0, cnt, r, gs, ngs, cs, ge, nge, rp, eu, pk;
    float scale;
};

// The slot records a CTA touches sit in a window of kSlotCache consecutive
// tiles from its first one (both of its lists are in slot order); the window
// is copied to shared memory in the prologue and tiles past it read the plan.
constexpr int kSlotCache = 32;

__device__ __forceinline__ Slot load_slot(const unsigned char *plan, int32_t a, const int4 *cache, int32_t base) {
    int4 v[4];
    const int4 *p = (a >= base && a < base + kSlotCache)
                        ? cache + 4 * (a - base)
                        : reinterpret_cast<const int4 *>(plan + plan_slots_off() + size_t(a) * sizeof(SlotRec));
    if (a >= base && a < base + kSlotCache) {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = p[q];
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = __ldcg(p + q);
    }
    Slot s;
    s.s = v[0].x;
    s.seg0 = v[0].y;
    s.cnt = v[0].z;
    s.r = v[0].w;
    s.scale = __int_as_float(v[1].x);
    s.gs = v[1].y;
    s.ngs = v[1].z;
    s.cs = v[1].w;
    s.ge = v[2].x;
    s.nge = v[2].y;
    s.rp = v[3].x;
    s.eu = v[3].y;
    s.pk = v[3].z;
    return s;
}


struct Ctx {
    int32_t T, n, k, r_max, nkb, ublk;
    int32_t off[LORA_MAX_SLICES + 1];
    const unsigned char *plan;
    const int32_t *ids;
    const unsigned char *maps;
};


// Expand unit u (0 <= u < ublk) of a token group -> slice and column block.
__device__ __forceinline__ void unit_slice(const Ctx &C, int32_t u, int32_t &i, int32_t &cb) {
    i = 0;
    while (true) {
        const int32_t nb = cdiv(C.off[i + 1] - C.off[i], kUnitCols);
        if (u < nb || i + 1 >= C.n) break;
        u -= nb;
        ++i;
    }
    cb = u;
}

// ---------------------------------------------------------------------------
// Tensor-core roles (tcgen05; warp 2 lane 0 issues, warps 2..5 read results)
// ---------------------------------------------------------------------------
// Adds v to a per-slot counter with release semantics: the sums this CTA
// added before (ordered by the barrier that precedes the call) are visible to
// whoever acquires the new count.
__device__ __forceinline__ void red_release_add(int32_t *p, int32_t v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Issues one shrink stage.  The stage holds the A rows of its nb k-blocks
// (nb * nr rows) and then their x tiles (nb * gpad rows), both K-major with the
// 128-byte swizzle; ranks go to tensor-memory lanes, tokens to columns.
//   n r <= 128: one MMA per K=16 step covers every k-block of the stage:
//     D[(kbl, rank)][(kbl', token)] (+)= A rows . x rows over the step's 16
//     columns of each row's own block; only the diagonal blocks kbl = kbl'
//     are products of matching columns, and the epilogue reads just those
//     (the plan keeps nb * nr <= 128 and nb * gpad <= 256).  Four MMAs per
//     stage however many k-blocks it holds.
//   n r > 128 (nb = 1): ranks 0..127 into columns 0.., ranks 128.. into
//     columns 128.. (a second MMA per step).
// `first`: the run's first stage, whose first step overwrites D.
__device__ __forceinline__ void shrink_mma_stage(uint32_t tmem, uint32_t sbase, int32_t nb, int32_t gpad, int32_t nr,
                                                 bool first) {
    const uint32_t xa = sbase + static_cast<uint32_t>(nb * nr) * 128u;
    const uint32_t idesc = tc::idesc_bf16(128, nb * gpad);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const bool acc = !(first && kk == 0);
        const uint64_t xd = tc::smem_desc(xa + 32 * kk, 1024, tc::kLayoutSW128);
        tc::mma_bf16(tmem, tc::smem_desc(sbase + 32 * kk, 1024, tc::kLayoutSW128), xd, idesc, acc);
        if (nr > 128)
            tc::mma_bf16(tmem + 128, tc::smem_desc(sbase + 128 * 128 + 32 * kk, 1024, tc::kLayoutSW128), xd, idesc,
                         acc);
    }
}

__device__ __forceinline__ void red_v4(float *p, float4 v) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1,%2,%3,%4};" :: "l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w) : "memory");
}

// Reads the run's D from tensor memory and adds it into the call's fp32 sums
// acc_buf[p][i * r_max + j].  This warp's 32 lanes are D rows lane_base +
// lane: for n r <= 128 row (kbl, rank) of the nbr k-blocks the run's stages
// held, whose tokens sit in columns kbl * gpad..; for n r > 128 rank
// 128 d + row of D_d.  Each 16-token load is turned around through the warp's
// 2 KB of scratch (shared memory) so that a lane adds four consecutive ranks of
// one token with one 16-byte add; rows holding the same rank for different
// k-blocks add into the same sums.
__device__ __forceinline__ void shrink_epilogue(const Ctx &C, const Slot &sl, int32_t p0, int32_t gsz, int32_t gpad,
                                                int32_t nbr, uint32_t tmem, int32_t lane_base, int32_t lane,
                                                float *acc_buf, float *scr) {
    const int32_t nr = C.n * sl.r, NC = C.n * C.r_max;
    const int32_t nd = nr > 128 ? 2 : 1, rows = nr > 128 ? nr : nbr * nr;
    const int32_t rg = lane & 7, tq = lane >> 3;  // after the turn: ranks 4 rg .. 4 rg + 3, tokens tq + 4 k
    for (int32_t d = 0; d < nd; ++d) {
        const int32_t row0 = 128 * d + lane_base;  // warp-uniform
        if (row0 >= rows) continue;
        // this lane's four rows after the turn (a group of four never crosses a
        // slice or a k-block: r and n r are multiples of 8)
        const int32_t grow = row0 + 4 * rg;
        const int32_t gkbl = nd == 2 ? 0 : grow / nr, grank = nd == 2 ? grow : grow - gkbl * nr;
        const int32_t gi = grank / sl.r, gj = grank - gi * sl.r;
        float *dst = acc_buf + static_cast<size_t>(p0) * NC + gi * C.r_max + gj;
        const int32_t kb0 = nd == 2 ? 0 : row0 / nr, kb1 = nd == 2 ? 0 : min(row0 + 31, rows - 1) / nr;
        for (int32_t kc = kb0; kc <= kb1; ++kc) {
            const bool mine = grow < rows && gkbl == kc;
            for (int32_t t0 = 0; t0 < gsz; t0 += 16) {
                uint32_t r[16];
                tc::tmem_ld16(tmem + (static_cast<uint32_t>(lane_base) << 16) +
                                  static_cast<uint32_t>(128 * d + kc * gpad + t0),
                              r);
#pragma unroll
                for (int e = 0; e < 16; ++e) scr[e * 32 + lane] = __uint_as_float(r[e]);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int32_t t = tq + 4 * k;
                    if (mine && t0 + t < gsz)
                        red_v4(dst + static_cast<size_t>(t0 + t) * NC,
                               *reinterpret_cast<const float4 *>(scr + t * 32 + 4 * rg));
                }
                __syncwarp();
            }
        }
    }
}

// Issues one expand unit: D[128 columns][gpad tokens] = B box [128][rp] x
// sums [gpad][rp]^T over the rank padded to 16 (K-major, swizzle by rp).
__device__ __forceinline__ void expand_mma_unit(uint32_t tmem_d, uint32_t bbox, uint32_t xbuf, int32_t rp, int32_t r,
                                                uint32_t idesc) {
    const uint32_t layout = tc::layout_for_rowb(static_cast<uint32_t>(rp * 2));
    const uint32_t sbo = static_cast<uint32_t>(16 * rp);  // 8 rows of rp ranks
    const int32_t ksteps = pad16i(r) >> 4;
    for (int32_t kk = 0; kk < ksteps; ++kk)
        tc::mma_bf16(tmem_d, tc::smem_desc(bbox + 32 * kk, sbo, layout), tc::smem_desc(xbuf + 32 * kk, sbo, layout),
                     idesc, kk > 0);
}

// One expand unit's epilogue, in shared memory: this warp's 32 lanes are
// output columns lane_base + lane of the unit; the y tile ([yrows][128] bf16,
// 256-byte rows) becomes y + s * acc rounded once to bf16, in place.  The rows
// go to global memory afterwards.
__device__ __forceinline__ void expand_epilogue(float scale, int32_t yrows, uint32_t tmem_d, unsigned char *ytile,
                                                int32_t lane_base, int32_t lane) {
    uint16_t *yc = reinterpret_cast<uint16_t *>(ytile) + lane_base + lane;
    for (int32_t t0 = 0; t0 < yrows; t0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(tmem_d + (static_cast<uint32_t>(lane_base) << 16) + static_cast<uint32_t>(t0), r);
        uint16_t yo[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) yo[e] = t0 + e < yrows ? yc[(t0 + e) * kUnitCols] : 0;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float v = bf16lo_to_f32(yo[e]) + scale * __uint_as_float(r[e]);
            if (t0 + e < yrows) yc[(t0 + e) * kUnitCols] = static_cast<uint16_t>(pack_bf16x2(v, 0.f));
        }
    }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2) tma_decode_kernel(const __grid_constant__ TArgs a) {
    extern __shared__ unsigned char smem_raw[];
    // full[kStages], empty[kStages], run_done, acc_full[2] (one per half of tensor memory)
    __shared__ __align__(8) uint64_t bars[2 * kStages + 3];
    __shared__ int32_t s_abort, s_flag;
    __shared__ uint32_t s_tmem;
    __shared__ int32_t s_rows[kGe];                      // token ids of the expand run's group (tensor-core warps)
    __shared__ int32_t s_xids[128];                      // token ids of the gather warp's current group
    __shared__ int4 s_slots[4 * kSlotCache];              // slot records of tiles [slot_base, + kSlotCache)

    pdl_launch_dependents();
    const PlanHdr *H = reinterpret_cast<const PlanHdr *>(a.plan);
    const int4 h0 = __ldcg(reinterpret_cast<const int4 *>(H)), h1 = __ldcg(reinterpret_cast<const int4 *>(H) + 1);
    const int4 h2 = __ldcg(reinterpret_cast<const int4 *>(H) + 2), h3 = __ldcg(reinterpret_cast<const int4 *>(H) + 3);
    const uint64_t table = __ldcg(&H->table);
    // the CTA's record in the same round trip (a plan buffer is at least
    // tma_plan_size(T, S) bytes, so the read is in bounds whatever it holds)
    const CtaRec *cr = reinterpret_cast<const CtaRec *>(a.plan + plan_ctas_off(a.S)) + blockIdx.x;
    const int4 crs = __ldcg(reinterpret_cast<const int4 *>(cr)), cre = __ldcg(reinterpret_cast<const int4 *>(cr) + 1);
    // h0 = magic, T, S, n; h1 = k, r_max, na, grid; h2 = off[0..3]; h3 = off[4], nkb, ublk, pad
    bool valid = h0.x == kPlanMagic && h0.y == a.T && h0.z == a.S && h0.w == a.n && h1.x == a.k &&
                 h1.y == a.r_max && h1.w == static_cast<int32_t>(gridDim.x) && table != 0;
    const int32_t offs[5] = {h2.x, h2.y, h2.z, h2.w, h3.x};
    for (int i = 0; i <= LORA_MAX_SLICES; ++i) valid = valid && offs[i] == a.off[i];
    if (!valid) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
        return;
    }
    Ctx C;
    C.T = a.T;
    C.n = a.n;
    C.k = a.k;
    C.r_max = a.r_max;
    C.nkb = h3.y;
    C.ublk = h3.z;
    for (int i = 0; i <= LORA_MAX_SLICES; ++i) C.off[i] = a.off[i];
    C.plan = a.plan;
    C.ids = reinterpret_cast<const int32_t *>(a.plan + plan_ids_off(a.S));
    C.maps = reinterpret_cast<const unsigned char *>(table) + TmaTableLayout(a.S, a.n).maps;

    const uint32_t ring = (sa(smem_raw) + 1023u) & ~1023u;
    const uint32_t xbuf = ring + kStages * kStageBytes;
    const uint32_t bar0 = sa(&bars[0]);  // full[st] at bar0 + 8 st, empty[st] at bar0 + 8 (kStages + st)
    const uint32_t bar_done = bar0 + 8 * (2 * kStages), bar_acc = bar_done + 8;
    const int32_t slot_base = min(crs.x, cre.x);
    const int32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    {
        const int32_t na = h1.z;
        const int32_t e = threadIdx.x;  // 128 int4: four per cached record
        if (e < 4 * kSlotCache && slot_base + (e >> 2) < na)
            s_slots[e] = __ldcg(reinterpret_cast<const int4 *>(a.plan + plan_slots_off() +
                                                                size_t(slot_base) * sizeof(SlotRec)) + e);
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(bar0 + 8 * st, 1 + 32);         // the producer's expect_tx + the 32 gather lanes
            mbar_init(bar0 + 8 * (kStages + st), 1);  // a tcgen05.commit, or the expand's last epilogue
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_acc, 1);
        mbar_init(bar_acc + 8, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_abort = 0;
    }
    if (warp == 2) tc::tmem_alloc(&s_tmem, kTmemCols);  // whole warp
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    volatile int32_t *abort = &s_abort;

    if (warp == 0) {
        // ---- TMA producer: adapter weights only, never waits for the previous grid
        if (lane == 0) {
            uint64_t policy;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
            uint32_t c = 0;
            int32_t tile = crs.x, idx = crs.y, left = crs.z, cur = -1;
            Slot sl{};
            while (left > 0 && !*abort) {
                if (tile != cur) {
                    sl = load_slot(C.plan, tile, s_slots, slot_base);
                    cur = tile;
                }
                const int32_t g = idx / C.nkb, kb = idx % C.nkb;
                const int32_t nb = min(min(sl.cs, C.nkb - kb), left);
                const int32_t gpad = pad16i(min(sl.gs, sl.cnt - g * sl.gs));
                const uint32_t st = c % kStages;
                if (c >= kStages && !ring_wait(bar0 + 8 * (kStages + st), ((c / kStages) + 1) & 1, abort, kCopyBackoffNs))
                    break;
                const uint32_t full = bar0 + 8 * st;
                const uint32_t dst = ring + st * kStageBytes;  // the A rows open the stage
                mbar_expect_tx(full, static_cast<uint32_t>(nb * C.n * sl.r) * 128u);
                const unsigned char *am = C.maps + static_cast<size_t>(sl.s) * (kMapsPerSlot * 128);
                if (sl.pk) {
                    // packed slices: blocks of depth 8, 4, 2, 1 (one copy each)
                    const int32_t nr = C.n * sl.r;
                    for (int32_t kbl = 0, d = 3; d >= 0; --d)
                        if (nb & (1 << d)) {
                            tma_load_3d(dst + static_cast<uint32_t>(kbl * nr) * 128u, am + d * 128, 0, 0, kb + kbl, full,
                                        policy);
                            kbl += 1 << d;
                        }
                } else {
                    for (int32_t kbl = 0; kbl < nb; ++kbl)
                        for (int32_t i = 0; i < C.n; ++i)
                            tma_load_3d(dst + static_cast<uint32_t>((kbl * C.n + i) * sl.r) * 128u, am + i * 128, 0, 0,
                                        kb + kbl, full, policy);
                }
                ++c;
                idx += nb;
                left -= nb;
                if (idx == sl.ngs * C.nkb) {
                    ++tile;
                    idx = 0;
                }
            }
            tile = cre.x;
            idx = cre.y;
            left = cre.z;
            cur = -1;
            while (left > 0 && !*abort) {
                if (tile != cur) {
                    sl = load_slot(C.plan, tile, s_slots, slot_base);
                    cur = tile;
                }
                int32_t i, cb;
                unit_slice(C, idx % C.ublk, i, cb);
                const int32_t m = min(sl.eu, min(cdiv(C.off[i + 1] - C.off[i], kUnitCols) - cb, left));
                const uint32_t st = c % kStages;
                if (c >= kStages && !ring_wait(bar0 + 8 * (kStages + st), ((c / kStages) + 1) & 1, abort, kCopyBackoffNs))
                    break;
                const uint32_t full = bar0 + 8 * st, bbox = static_cast<uint32_t>(kUnitCols * sl.rp * 2);
                mbar_expect_tx(full, static_cast<uint32_t>(m) * bbox);
                for (int32_t u = 0; u < m; ++u)
                    tma_load_2d(ring + st * kStageBytes + u * bbox,
                                C.maps + static_cast<size_t>(sl.s) * (kMapsPerSlot * 128) + (4 + i) * 128, 0,
                                (cb + u) * kUnitCols,
                                full, policy);
                ++c;
                idx += m;
                left -= m;
                if (idx == sl.nge * C.ublk) {
                    ++tile;
                    idx = 0;
                }
            }
        }
    } else if (warp == 1) {
        // ---- row gathers through the tensor maps of x and y, four token rows
        // per copy (lane l copies rows 4 l .. 4 l + 3 of the group); the ids of
        // the current group are staged in shared memory
        pdl_wait();
        uint32_t c = 0;
        int32_t tile = crs.x, idx = crs.y, left = crs.z, cur = -1, cur_g = -1;
        Slot sl{};
        while (left > 0 && !__any_sync(0xffffffffu, *abort != 0)) {
            if (tile != cur) {
                sl = load_slot(C.plan, tile, s_slots, slot_base);
                cur = tile;
                cur_g = -1;
            }
            const int32_t g = idx / C.nkb, kb = idx % C.nkb;
            const int32_t nb = min(min(sl.cs, C.nkb - kb), left);
            const int32_t gsz = min(sl.gs, sl.cnt - g * sl.gs), gpad = pad16i(gsz), nq = (gsz + 3) >> 2;
            if (g != cur_g) {
                __syncwarp();
                for (int32_t r = lane; r < gsz; r += 32) {
                    const int32_t p = __ldcg(C.ids + sl.seg0 + g * sl.gs + r);
                    s_xids[r] = a.xdiv == 1 ? p : p / a.xdiv;
                }
                __syncwarp();
                cur_g = g;
            }
            const uint32_t st = c % kStages;
            const bool free_ = c < kStages || ring_wait(bar0 + 8 * (kStages + st), ((c / kStages) + 1) & 1, abort,
                                                        kCopyBackoffNs);
            if (__any_sync(0xffffffffu, !free_)) break;
            const uint32_t full = bar0 + 8 * st;
            if (lane == 0)
                mbar_expect_tx(full, static_cast<uint32_t>(nb * nq) * 512u);
            else
                mbar_arrive(full);
            __syncwarp();
            if (lane < nq) {
                // x rows after the stage's A rows: [nb][gpad][64] bf16, 128-byte swizzle
                const int4 rows = four_ids(s_xids, lane, gsz);
                const uint32_t xdst = ring + st * kStageBytes + static_cast<uint32_t>(nb * sl.r * C.n) * 128u +
                                      static_cast<uint32_t>(lane) * 512u;
                for (int32_t kbl = 0; kbl < nb; ++kbl)
                    tma_gather4(xdst + static_cast<uint32_t>(kbl * gpad) * 128u, &a.xmap, (kb + kbl) * 64, rows, full);
            }
            ++c;
            idx += nb;
            left -= nb;
            if (idx == sl.ngs * C.nkb) {
                ++tile;
                idx = 0;
            }
        }
        tile = cre.x;
        idx = cre.y;
        left = cre.z;
        cur = -1;
        cur_g = -1;
        while (left > 0 && !__any_sync(0xffffffffu, *abort != 0)) {
            if (tile != cur) {
                sl = load_slot(C.plan, tile, s_slots, slot_base);
                cur = tile;
                cur_g = -1;
            }
            const int32_t g = idx / C.ublk;
            int32_t i, cb;
            unit_slice(C, idx % C.ublk, i, cb);
            const int32_t gsz = min(sl.ge, sl.cnt - g * sl.ge);
            if (g != cur_g) {
                __syncwarp();
                for (int32_t r = lane; r < gsz; r += 32) s_xids[r] = __ldcg(C.ids + sl.seg0 + g * sl.ge + r);
                __syncwarp();
                cur_g = g;
            }
            const int32_t di = C.off[i + 1] - C.off[i];
            const int32_t m = min(sl.eu, min(cdiv(di, kUnitCols) - cb, left));
            const uint32_t st = c % kStages;
            const bool free_ = c < kStages || ring_wait(bar0 + 8 * (kStages + st), ((c / kStages) + 1) & 1, abort,
                                                        kCopyBackoffNs);
            if (__any_sync(0xffffffffu, !free_)) break;
            // y rows after the m B boxes: [m][gsz rounded to 8][128] bf16, 256-byte rows, 16-byte
            // copies (a warp's 32 copies cover two rows); rows past the group are zeros
            const uint32_t ydst = ring + st * kStageBytes + static_cast<uint32_t>(m * kUnitCols * sl.rp * 2);
            const int32_t yrows = ytile_rows(gsz);
            for (int32_t u = 0; u < m; ++u)
                for (int32_t e = lane; e < yrows * 16; e += 32) {
                    const int32_t row = e >> 4, ch = e & 15, col = (cb + u) * kUnitCols + ch * 8;
                    const bool v = row < gsz && col < di;
                    cp16(ydst + static_cast<uint32_t>(u * yrows * 256 + e * 16),
                         a.y + static_cast<int64_t>(s_xids[v ? row : 0]) * a.ldy + C.off[i] + (v ? col : 0), v);
                }
            cp_arrive_noinc(bar0 + 8 * st);
            ++c;
            idx += m;
            left -= m;
            if (idx == sl.nge * C.ublk) {
                ++tile;
                idx = 0;
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // ---- tensor-core group: warps 2..5 (warp w reads tensor-memory lanes
        // 32 (w % 4) ..); warp 2 lane 0 issues every tcgen05 instruction
        pdl_wait();
        const int32_t mtid = threadIdx.x - 64, lane_base = 32 * (warp & 3);
        const bool issuer = warp == 2 && lane == 0;
        const int32_t gen = __ldcg(a.gen);
        float *acc_buf = (gen & 1) ? a.acc1 : a.acc0;
        int32_t *done = (gen & 1) ? a.done1 : a.done0;
        {
            // clear the set the previous call used (the next call adds into it)
            float *other = (gen & 1) ? a.acc0 : a.acc1;
            int32_t *odone = (gen & 1) ? a.done0 : a.done1;
            const size_t total4 = (static_cast<size_t>(C.n) * C.T * C.r_max) / 4;
            const size_t per = (total4 + gridDim.x - 1) / gridDim.x;
            const size_t lo = per * blockIdx.x, hi = min(total4, lo + per);
            for (size_t e = lo + mtid; e < hi; e += kMmaThreads)
                reinterpret_cast<float4 *>(other)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int32_t s = blockIdx.x * kMmaThreads + mtid; s < a.S; s += gridDim.x * kMmaThreads) odone[s] = 0;
        }
        // the shrink epilogue's scratch: 2 KB per warp in the expand's sum tile,
        // which no expand run uses before this CTA's last shrink run
        float *xscr = reinterpret_cast<float *>(smem_raw + (xbuf - sa(smem_raw))) + (warp & 3) * 512;
        uint32_t c = 0, runs = 0, units = 0;
        bool fail = false;  // the same in all four warps: every change of it goes through mma_any
        int32_t tile = crs.x, idx = crs.y, left = crs.z;
        while (left > 0 && !fail) {
            const Slot sl = load_slot(C.plan, tile, s_slots, slot_base);
            const int32_t g = idx / C.nkb, kb = idx % C.nkb;
            const int32_t run_len = min(C.nkb - kb, left);
            const int32_t nr = C.n * sl.r, gsz = min(sl.gs, sl.cnt - g * sl.gs), gpad = pad16i(gsz);
            const int32_t nst = cdiv(run_len, sl.cs);  // the run's stages (the copy warps split it the same way)
            bool bad = false;
            if (issuer) {
                for (int32_t q = 0, dp = 0; q < nst; ++q) {
                    const int32_t nb = min(sl.cs, run_len - dp);
                    const uint32_t st = (c + q) % kStages;
                    if (!ring_wait(bar0 + 8 * st, ((c + q) / kStages) & 1, abort)) {
                        bad = true;
                        break;
                    }
                    tc::fence_after_sync();
                    shrink_mma_stage(tmem, ring + st * kStageBytes, nb, gpad, nr, q == 0);
                    tc::mma_commit(reinterpret_cast<uint64_t *>(&bars[kStages + st]));  // frees the stage
                    dp += nb;
                }
                tc::mma_commit(reinterpret_cast<uint64_t *>(&bars[2 * kStages]));  // the run's D is complete
            }
            __syncwarp();
            c += nst;
            const bool got = __all_sync(0xffffffffu, ring_wait(bar_done, runs & 1, abort));  // tcgen05.ld: whole warps
            ++runs;
            if (got) {
                tc::fence_after_sync();
                shrink_epilogue(C, sl, sl.seg0 + g * sl.gs, gsz, gpad, min(sl.cs, run_len), tmem, lane_base, lane,
                                acc_buf, xscr);
            }
            tc::fence_before_sync();
            // every warp's sums of the run are issued and D may be overwritten
            fail = mma_any(bad || !got);
            if (fail) break;
            if (mtid == 0) red_release_add(done + sl.s, run_len);
            idx += run_len;
            left -= run_len;
            if (idx == sl.ngs * C.nkb) {
                ++tile;
                idx = 0;
            }
        }
        tile = cre.x;
        idx = cre.y;
        left = cre.z;
        while (left > 0 && !fail) {
            const Slot sl = load_slot(C.plan, tile, s_slots, slot_base);
            const int32_t g = idx / C.ublk;
            int32_t i, cb;
            unit_slice(C, idx % C.ublk, i, cb);
            const int32_t blocks_i = cdiv(C.off[i + 1] - C.off[i], kUnitCols);
            const int32_t run_len = min(blocks_i - cb, left);
            const int32_t gsz = min(sl.ge, sl.cnt - g * sl.ge), gpad = pad16i(gsz);
            const int32_t p0 = sl.seg0 + g * sl.ge;
            const int32_t r16 = pad16i(sl.r), rp = sl.rp;
            // the slot's sums are complete once every k-block of every group is in
            if (mtid == 0) {
                const int32_t need = sl.ngs * C.nkb;
                int32_t ok = *abort ? -1 : 1;
                if (ok > 0 && ld_acquire(done + sl.s) < need) {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire(done + sl.s) < need) {
                        if (globaltimer_ns() - t0 > kSlotLimitNs) {
                            report_error(a.err, LORA_ERR_TIMEOUT);
                            ok = 0;
                            break;
                        }
                        __nanosleep(100);
                    }
                }
                s_flag = ok;
            }
            mma_barrier();
            const int32_t flag = s_flag;
            if (flag < 0) {  // the ring has given up
                fail = true;
                break;
            }
            const bool ok = flag != 0;  // false: the slot's y rows stay as they are, its stages still drain
            if (ok) {
                // the group's sums -> bf16 [gpad][rp] tile with the swizzle of rp-rank rows
                // (rows past the group repeat its last token; their results are never
                // stored); every load of a thread is issued before its first store
                if (mtid < gsz) s_rows[mtid] = __ldcg(C.ids + p0 + mtid);
                const int32_t pairs = r16 >> 1, total = gpad * pairs, NC = C.n * C.r_max;
                constexpr int kPer = kGe * 32 / kMmaThreads;
                float2 v[kPer];
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int32_t e = mtid + u * kMmaThreads;
                    const int32_t row = e / pairs, j = 2 * (e - row * pairs);
                    v[u] = make_float2(0.f, 0.f);
                    if (e < total && j < sl.r)
                        v[u] = __ldcg(reinterpret_cast<const float2 *>(
                            acc_buf + static_cast<size_t>(p0 + min(row, gsz - 1)) * NC + i * C.r_max + j));
                }
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int32_t e = mtid + u * kMmaThreads;
                    const int32_t row = e / pairs, j = 2 * (e - row * pairs);
                    if (e < total)
                        sts32(xbuf + tc::swz_offset(row, j >> 3, rp * 2) + static_cast<uint32_t>((j & 7) * 2),
                              pack_bf16x2(v[u].x, v[u].y));
                }
                tc::fence_async_smem();  // the tile is read by the tensor cores (async proxy)
            }
            mma_barrier();
            const uint32_t idesc = tc::idesc_bf16(128, gpad);
            const uint32_t bbox = static_cast<uint32_t>(kUnitCols * rp * 2);
            const int32_t di = C.off[i + 1] - C.off[i], yrows = ytile_rows(gsz);
            const int32_t nstg = cdiv(run_len, sl.eu);
            // Stage j of the run puts its m units' D in tensor-memory half (units + j) & 1
            // (unit u at column u gpad of the half) and commits to acc_full of that half.
            // The issuing thread starts stage j + 1's MMAs before stage j's epilogue
            // when j + 1's data is already in, so the tensor cores overlap the
            // epilogue and the stores.
            int32_t issued = 0;  // stages whose MMAs are issued (issuing thread only)
            auto issue_stage = [&](int32_t j) {
                const uint32_t sb = ring + ((c + j) % kStages) * kStageBytes;
                const int32_t mj = min(sl.eu, run_len - j * sl.eu);
                const uint32_t half = static_cast<uint32_t>((units + j) & 1) * 128u;
                for (int32_t u = 0; u < mj; ++u)
                    expand_mma_unit(tmem + half + static_cast<uint32_t>(u * gpad), sb + u * bbox, xbuf, rp, sl.r, idesc);
                tc::mma_commit(reinterpret_cast<uint64_t *>(&bars[2 * kStages + 1 + ((units + j) & 1)]));
            };
            for (int32_t j = 0; j < nstg && !fail; ++j) {
                const int32_t u0 = j * sl.eu, m = min(sl.eu, run_len - u0);
                const uint32_t st = (c + j) % kStages, sbase = ring + st * kStageBytes;
                fail = mma_any(!ring_wait(bar0 + 8 * st, ((c + j) / kStages) & 1, abort));
                if (fail) break;
                tc::fence_after_sync();
                if (ok && issuer) {
                    if (issued == j) issue_stage(issued++);
                    if (issued == j + 1 && j + 1 < nstg &&
                        mbar_try_wait(bar0 + 8 * ((c + j + 1) % kStages), ((c + j + 1) / kStages) & 1)) {
                        tc::fence_after_sync();
                        issue_stage(issued++);
                    }
                }
                __syncwarp();
                bool got = true;
                const uint32_t yt0 = sbase + static_cast<uint32_t>(m) * bbox;
                if (ok) {
                    const uint32_t U = units + j, half = (U & 1) * 128u;
                    got = __all_sync(0xffffffffu, ring_wait(bar_acc + 8 * (U & 1), (U >> 1) & 1, abort));
                    if (got) {
                        tc::fence_after_sync();
                        for (int32_t u = 0; u < m; ++u)
                            expand_epilogue(sl.scale, yrows, tmem + half + static_cast<uint32_t>(u * gpad),
                                            smem_raw + (yt0 + static_cast<uint32_t>(u * yrows * 256) - sa(smem_raw)),
                                            lane_base, lane);
                    }
                }
                tc::fence_before_sync();
                // the tiles' rows are final and this half of tensor memory may be refilled
                fail = mma_any(!got);
                if (fail) break;
                if (ok) {
                    // the rows to global memory: 16-byte pieces, a row's 16 pieces by consecutive threads
                    for (int32_t u = 0; u < m; ++u) {
                        const int32_t col0 = (cb + u0 + u) * kUnitCols;
                        const int32_t nch = min(kUnitCols, di - col0) >> 3;
                        const uint32_t yt = yt0 + static_cast<uint32_t>(u * yrows * 256);
                        for (int32_t e = mtid; e < gsz * 16; e += kMmaThreads) {
                            const int32_t row = e >> 4, ch = e & 15;
                            if (ch < nch)
                                stg128(a.y + static_cast<int64_t>(s_rows[row]) * a.ldy + C.off[i] + col0 + ch * 8,
                                       lds128(yt + static_cast<uint32_t>(row * 256 + ch * 16)));
                        }
                    }
                }
                mma_barrier();  // every read of the stage is done
                if (mtid == 0) mbar_arrive(bar0 + 8 * (kStages + st));
            }
            if (fail) break;
            c += nstg;
            if (ok) units += nstg;
            idx += run_len;
            left -= run_len;
            if (idx == sl.nge * C.ublk) {
                ++tile;
                idx = 0;
            }
        }
        if (fail && mtid == 0) *abort = 1;
    }

    tc::fence_before_sync();
    __syncthreads();
    const bool aborted = *abort != 0;  // nobody writes it past the barrier
    if (aborted) {
        // copies and MMAs that a stalled ring may still have in flight end
        // within microseconds; wait well past that before the shared and
        // tensor memory are given back
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
    }
    if (warp == 2) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0) {
        if (aborted) report_error(a.err, LORA_ERR_TIMEOUT);
        pdl_wait();
        __threadfence();
        if (atomicAdd(a.exits, 1) == static_cast<int32_t>(gridDim.x) - 1) {
            atomicExch(a.exits, 0);
            atomicAdd(a.gen, 1);
        }
    }
}

// ---------------------------------------------------------------------------
// Plan builder: one CTA per slot table (job)
// ---------------------------------------------------------------------------
constexpr int kMaxPlanJobs = 120;
struct TmaPlanJobs {
    const void *table[kMaxPlanJobs];
    unsigned char *plan[kMaxPlanJobs];
};

struct PArgs {
    const int32_t *sorted_ids, *seg, *active;
    int32_t *err;
    int32_t T, grid;
};

// Largest t in [0, N) with pref[t] <= v (pref ascending, pref[0] <= v).
__device__ __forceinline__ int32_t last_le64(const int64_t *pref, int32_t N, int64_t v) {
    int32_t lo = 0, hi = N;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (pref[mid] <= v) lo = mid + 1;
        else hi = mid;
    }
    return lo - 1;
}

// Global index of the first piece whose weight start is >= v: tiles t hold
// P[t] = ppref[t + 1] - ppref[t] pieces of equal weight w[t].
__device__ __forceinline__ int32_t piece_at(const int64_t *wpref, const int32_t *ppref, const int32_t *w, int32_t N,
                                            int64_t v) {
    if (N == 0 || v >= wpref[N]) return N == 0 ? 0 : ppref[N];
    const int32_t t = last_le64(wpref, N, v);
    const int64_t i = (v - wpref[t] + w[t] - 1) / w[t];
    return ppref[t] + static_cast<int32_t>(i);
}

__device__ __forceinline__ void locate(const int32_t *ppref, int32_t N, int32_t gidx, int32_t &tile, int32_t &idx) {
    if (gidx >= ppref[N]) {
        tile = N;
        idx = 0;
        return;
    }
    int32_t lo = 0, hi = N;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (ppref[mid] <= gidx) lo = mid + 1;
        else hi = mid;
    }
    tile = lo - 1;
    idx = gidx - ppref[tile];
}

__global__ void __launch_bounds__(512) tma_plan_kernel(PArgs pa, Shape sh, TmaPlanJobs jobs) {
    extern __shared__ __align__(16) unsigned char psmem[];
    const int32_t S = sh.S;
    int32_t *flag = reinterpret_cast<int32_t *>(psmem);           // [S + 1]: valid, then compacted index
    int32_t *wps = flag + (S + 1);                                 // [S + 1] shrink piece weight
    int32_t *wpe = wps + (S + 1);                                  // [S + 1] expand unit weight
    int32_t *pps = wpe + (S + 1);                                  // [S + 1] shrink piece prefix
    int32_t *ppe = pps + (S + 1);                                  // [S + 1] expand unit prefix
    int32_t *scr = ppe + (S + 1);                                  // [48] scan scratch
    int64_t *wprs = reinterpret_cast<int64_t *>(psmem + (((6 * (S + 1) + 48) * 4 + 15) & ~15));  // [S + 1]
    int64_t *wpre = wprs + (S + 1);                                                               // [S + 1]
    __shared__ int32_t s_ok, s_na;

    const void *table = jobs.table[blockIdx.x];
    unsigned char *plan = jobs.plan[blockIdx.x];
    const int32_t *hdr = static_cast<const int32_t *>(table);
    const TableView tab(table, S, sh.n);
    const int32_t *mh = reinterpret_cast<const int32_t *>(static_cast<const char *>(table) + TmaTableLayout(S, sh.n).hdr);
    const int32_t *tflags =
        reinterpret_cast<const int32_t *>(static_cast<const char *>(table) + TmaTableLayout(S, sh.n).flags);
    const int32_t n = sh.n, nkb = sh.k / 64;
    int32_t ublk = 0;
    for (int i = 0; i < n; ++i) ublk += cdiv(sh.off[i + 1] - sh.off[i], kUnitCols);
    if (threadIdx.x == 0) {
        // the maps block is read only once the header says the table has one
        bool ok = hdr[0] == kTableMagic && hdr[1] == S && hdr[2] == n && (hdr[3] & kTableMapsFlag) != 0 &&
                  pa.seg[S + 1] == pa.T;
        ok = ok && mh[0] == kTmaTableMagic && mh[1] == S && mh[2] == n && mh[3] == sh.k;
        for (int i = 0; i <= LORA_MAX_SLICES; ++i) ok = ok && mh[4 + i] == sh.off[i];
        const int32_t na = pa.active[0];
        ok = ok && na >= 0 && na <= S;
        if (!ok) report_error(pa.err, LORA_ERR_INVALID_ARG);
        s_ok = ok;
        s_na = ok ? na : 0;
    }
    __syncthreads();
    PlanHdr *H = reinterpret_cast<PlanHdr *>(plan);
    if (!s_ok) {
        if (threadIdx.x == 0) H->magic = 0;  // a call with this plan refuses it
        return;
    }
    const int32_t na = s_na;
    // valid active slots: rank in (0, min(r_max, 64)], n * r <= 192, tokens > 0
    for (int32_t e = threadIdx.x; e < S; e += blockDim.x) {
        int32_t v = 0;
        if (e < na) {
            const int32_t s = pa.active[1 + e];
            if (s >= 0 && s < S) {
                const int32_t r = tab.rank[s], cnt = pa.seg[s + 1] - pa.seg[s];
                const bool rank_ok = r > 0 && r <= sh.r_max && r <= kMaxRank && n * r <= kMaxNR && r % 8 == 0;
                if (r > 0 && !rank_ok) report_error(pa.err, LORA_ERR_RANK);
                v = rank_ok && cnt > 0 ? 1 : 0;
            }
        }
        flag[e] = v;
    }
    __syncthreads();
    const int32_t nv = block_exclusive_scan(flag, S, scr);  // flag[e] = compacted index of active entry e
    SlotRec *recs = reinterpret_cast<SlotRec *>(plan + plan_slots_off());
    for (int32_t e = threadIdx.x; e < na; e += blockDim.x) {
        const int32_t s = pa.active[1 + e];
        if (s < 0 || s >= S) continue;
        const int32_t r = tab.rank[s], cnt = pa.seg[s + 1] - pa.seg[s];
        const bool use = r > 0 && r <= sh.r_max && r <= kMaxRank && n * r <= kMaxNR && r % 8 == 0 && cnt > 0;
        if (!use) continue;
        const int32_t a = flag[e];
        const int32_t nr = n * r;
        const int32_t gmax = nr <= 96 ? 128 : 64;
        const int32_t ngs = cdiv(cnt, gmax), gs = cdiv(cnt, ngs);
        // k-blocks per stage: the A and x rows fit the stage's 256 rows; one MMA
        // covers the stage (nb n r <= 128 D rows, nb gpad <= 256 columns); at
        // most 15 (a packed stage is copied as blocks of 8, 4, 2 and 1)
        const int32_t cs = nr > 128 ? 1
                                    : max(1, min(min(min(nkb, 256 / (nr + pad16i(gs))), 128 / nr),
                                                 min(256 / pad16i(gs), 15)));
        const int32_t nge = cdiv(cnt, kGe), ge = cdiv(cnt, nge);
        SlotRec rec;
        rec.s = s;
        rec.seg0 = pa.seg[s];
        rec.cnt = cnt;
        rec.r = r;
        rec.scale = tab.scale[s];
        rec.gs = gs;
        rec.ngs = ngs;
        rec.cs = cs;
        rec.ge = ge;
        rec.nge = nge;
        // weights in 16-byte units: the bytes a piece moves plus the fixed costs
        // that bound small pieces (a four-row gather of x, an expand unit's
        // share of its stage's tensor-core round trip, epilogue and barriers)
        // A and x rows of one k-block, plus its share of the stage's fixed cost
        rec.wps = (nr + gs) * 8 + kGatherCost * ((gs + 3) >> 2) + kShrinkStageCost / cs;
        rec.wpe = 16 * r + 32 * ge + kUnitCost;                   // B tile [128][r], y rows read + written
        rec.rp = b_box_ranks(r);
        // as many 128-column units of one run per stage as fit: the B boxes and
        // their y rows (ge rounded up to 8) in the stage, their D in half of tensor memory
        rec.eu = max(1, min(kStageBytes / (kUnitCols * rec.rp * 2 + ytile_rows(ge) * kUnitCols * 2),
                            (kTmemCols / 2) / pad16i(ge)));
        rec.pk = (tflags[s] & kSlotPackedA) != 0;
        rec.pad = 0;
        recs[a] = rec;
        wps[a] = rec.wps;
        wpe[a] = rec.wpe;
        pps[a] = ngs * nkb;
        ppe[a] = nge * ublk;
    }
    __syncthreads();
    // prefixes: pieces (int32) and weights (int64)
    for (int32_t e = threadIdx.x; e <= S; e += blockDim.x) {
        if (e >= nv) {
            pps[e] = 0;
            ppe[e] = 0;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t acs = 0, ace = 0;
        int32_t cps = 0, cpe = 0;
        for (int32_t t = 0; t < nv; ++t) {
            wprs[t] = acs;
            wpre[t] = ace;
            acs += static_cast<int64_t>(wps[t]) * pps[t];
            ace += static_cast<int64_t>(wpe[t]) * ppe[t];
            const int32_t ps = pps[t], pe = ppe[t];
            pps[t] = cps;
            ppe[t] = cpe;
            cps += ps;
            cpe += pe;
        }
        wprs[nv] = acs;
        wpre[nv] = ace;
        pps[nv] = cps;
        ppe[nv] = cpe;
    }
    __syncthreads();
    CtaRec *ctas = reinterpret_cast<CtaRec *>(plan + plan_ctas_off(S));
    const int64_t G = pa.grid;
    for (int32_t b = threadIdx.x; b < pa.grid; b += blockDim.x) {
        CtaRec cr;
        {
            const int64_t W = wprs[nv];
            const int32_t f = piece_at(wprs, pps, wps, nv, (W * b + G - 1) / G);
            const int32_t l = piece_at(wprs, pps, wps, nv, (W * (b + 1) + G - 1) / G);
            locate(pps, nv, f, cr.s_tile, cr.s_idx);
            cr.s_count = l - f;
        }
        {
            const int64_t W = wpre[nv];
            const int32_t f = piece_at(wpre, ppe, wpe, nv, (W * b + G - 1) / G);
            const int32_t l = piece_at(wpre, ppe, wpe, nv, (W * (b + 1) + G - 1) / G);
            locate(ppe, nv, f, cr.e_tile, cr.e_idx);
            cr.e_count = l - f;
        }
        cr.pad0 = cr.pad1 = 0;
        ctas[b] = cr;
    }
    int32_t *ids = reinterpret_cast<int32_t *>(plan + plan_ids_off(S));
    for (int32_t p = threadIdx.x; p < pa.T; p += blockDim.x) ids[p] = pa.sorted_ids[p];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        PlanHdr h;
        memset(&h, 0, sizeof h);
        h.magic = kPlanMagic;
        h.T = pa.T;
        h.S = S;
        h.n = n;
        h.k = sh.k;
        h.r_max = sh.r_max;
        h.na = nv;
        h.grid = pa.grid;
        for (int i = 0; i <= LORA_MAX_SLICES; ++i) h.off[i] = sh.off[i];
        h.nkb = nkb;
        h.ublk = ublk;
        h.table = reinterpret_cast<uint64_t>(table);
        *H = h;
        __threadfence();
    }
}

size_t tma_plan_smem(int32_t S) { return (((6 * (S + 1) + 48) * 4 + 15) & ~size_t(15)) + 2 * 8 * size_t(S + 1); }

int num_sms_now(int &num_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
}

// The grid of one call: kCtasPerSm CTAs per SM of the current device.
int tma_grid_now(int &grid) {
    int num_sms = 0;
    const int e = num_sms_now(num_sms);
    grid = num_sms * kCtasPerSm;
    return e;
}

// ---------------------------------------------------------------------------
// Host: tensor-map encoding through the driver entry point (no libcuda link)
// ---------------------------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = []() -> EncodeTiled {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

}  // namespace

// A tensor map of a bf16 matrix of `rows` rows of `cols` elements, `ld`
// elements apart, read in boxes of box_rows x box_cols (box_cols * 2 bytes at
// most 128 with the 128-byte swizzle); false if the driver's encoder is
// unavailable or rejects the map.
bool encode_bf16_rows_map(CUtensorMap *m, const void *base, int64_t ld, int32_t rows, int32_t cols, int32_t box_rows,
                          int32_t box_cols, bool swizzle128) {
    EncodeTiled enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t str[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t one[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, str, box, one,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Entry points used by lora_abi.cu
// ---------------------------------------------------------------------------
size_t tma_table_bytes(int32_t S, int32_t n) { return TmaTableLayout(S, n).bytes; }

// Fills the tensor-map block of a packed table in host memory (the ordinary
// part already packed).  Returns false when the driver's encoder is missing
// or rejects a map.
bool encode_tma_table(void *host_buf, const Shape &sh, const int32_t *ranks, const uint64_t *A_ptrs,
                      const uint64_t *B_ptrs) {
    const TmaTableLayout L(sh.S, sh.n);
    char *p = static_cast<char *>(host_buf);
    std::memset(p + L.hdr, 0, L.bytes - L.hdr);
    EncodeTiled enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint32_t one[3] = {1, 1, 1};
    // rows x k matrix at `base` viewed as [k / 64][rows][64]: the block index is
    // the outer dimension with a 128-byte stride, rows stride k * 2 bytes
    auto encode_a = [&](CUtensorMap *m, uint64_t base, int32_t rows, int32_t depth) {
        const cuuint64_t dim[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(sh.k / 64)};
        const cuuint64_t str[2] = {static_cast<cuuint64_t>(sh.k) * 2, 128};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(depth)};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, reinterpret_cast<void *>(base), dim, str, box, one,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    int32_t *flags = reinterpret_cast<int32_t *>(p + L.flags);
    for (int32_t s = 0; s < sh.S; ++s) {
        const int32_t r = ranks[s];
        if (r <= 0 || r > 256) continue;
        CUtensorMap *maps = reinterpret_cast<CUtensorMap *>(p + L.maps + size_t(s) * kMapsPerSlot * 128);
        const uint64_t a0 = A_ptrs[size_t(s) * sh.n];
        const uint64_t slice_bytes = uint64_t(r) * uint64_t(sh.k) * 2;
        bool packed = sh.n * r <= 256;
        for (int32_t i = 1; i < sh.n; ++i) packed = packed && A_ptrs[size_t(s) * sh.n + i] == a0 + i * slice_bytes;
        if (packed) {
            flags[s] = kSlotPackedA;
            for (int d = 0; d < 4; ++d)
                if (!encode_a(maps + d, a0, sh.n * r, 1 << d)) return false;
        } else {
            for (int32_t i = 0; i < sh.n; ++i)
                if (!encode_a(maps + i, A_ptrs[size_t(s) * sh.n + i], r, 1)) return false;
        }
        for (int32_t i = 0; i < sh.n; ++i) {
            const int32_t di = sh.off[i + 1] - sh.off[i];
            const cuuint64_t bdim[2] = {static_cast<cuuint64_t>(r), static_cast<cuuint64_t>(di)};
            const cuuint64_t bstr[1] = {static_cast<cuuint64_t>(r) * 2};
            const int32_t rp = b_box_ranks(r);
            const cuuint32_t bbox[2] = {static_cast<cuuint32_t>(rp), static_cast<cuuint32_t>(kUnitCols)};
            const CUtensorMapSwizzle bsw = rp == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                    : (rp == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
            if (enc(maps + 4 + i, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, reinterpret_cast<void *>(B_ptrs[s * sh.n + i]),
                    bdim, bstr, bbox, one, CU_TENSOR_MAP_INTERLEAVE_NONE, bsw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return false;
        }
    }
    reinterpret_cast<int32_t *>(p)[3] |= kTableMapsFlag;
    int32_t *mh = reinterpret_cast<int32_t *>(p + L.hdr);
    mh[0] = kTmaTableMagic;
    mh[1] = sh.S;
    mh[2] = sh.n;
    mh[3] = sh.k;
    for (int i = 0; i <= LORA_MAX_SLICES; ++i) mh[4 + i] = sh.off[i];
    return true;
}

bool decode_tma_supported(int32_t T, const Shape &sh) {
    return T >= 1 && T <= (1 << 20) && sh.r_max <= kMaxRank && sh.n * sh.r_max <= kMaxNR && sh.k % 64 == 0 &&
           tma_plan_smem(sh.S) <= 200 * 1024;
}

size_t tma_plan_bytes(int32_t T, const Shape &sh) { return plan_total(T, sh.S); }

cudaError_t launch_tma_plans(const Shape &sh, const void *const *tables, unsigned char *const *plans, int32_t count,
                             const int32_t *sorted_ids, const int32_t *seg, const int32_t *active, int32_t T,
                             int32_t *err, cudaStream_t stream) {
    if (!decode_tma_supported(T, sh)) return cudaErrorNotSupported;
    int grid = 0;
    cudaError_t e = static_cast<cudaError_t>(tma_grid_now(grid));
    if (e != cudaSuccess) return e;
    if (grid > kMaxGrid) return cudaErrorNotSupported;
    PArgs pa{sorted_ids, seg, active, err, T, grid};
    const size_t smem = tma_plan_smem(sh.S);
    e = cudaFuncSetAttribute(tma_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    for (int32_t j0 = 0; j0 < count; j0 += kMaxPlanJobs) {
        TmaPlanJobs jobs = {};
        const int32_t m = std::min(kMaxPlanJobs, count - j0);
        for (int32_t j = 0; j < m; ++j) {
            jobs.table[j] = tables[j0 + j];
            jobs.plan[j] = plans[j0 + j];
        }
        tma_plan_kernel<<<m, 512, smem, stream>>>(pa, sh, jobs);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// One call from a plan; ws_ctrl: [2 S] counters then gen, exits; acc0 / acc1:
// the two fp32 sum sets of [T][n r_max].
cudaError_t launch_tma_decode(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                              const unsigned char *plan, float *acc0, float *acc1, int32_t *ctrl, int32_t T,
                              int32_t *err, cudaStream_t stream, int32_t xdiv) {
    if (xdiv < 1 || T % xdiv != 0) return cudaErrorInvalidValue;
    if (!decode_tma_supported(T, sh)) return cudaErrorNotSupported;
    int grid = 0;
    cudaError_t e = static_cast<cudaError_t>(tma_grid_now(grid));
    if (e != cudaSuccess) return e;
    if (grid > kMaxGrid) return cudaErrorNotSupported;
    EncodeTiled enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    TArgs a;
    memset(&a, 0, sizeof a);
    {
        // x: [T][k] rows of ldx elements, box [1][64], 128-byte swizzle (the shrink's x tiles)
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(sh.k), static_cast<cuuint64_t>(T / xdiv)};
        const cuuint64_t str[1] = {static_cast<cuuint64_t>(ldx) * 2};
        const cuuint32_t box[2] = {64, 1}, one[2] = {1, 1};
        if (enc(&a.xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, str, box, one,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    a.x = x;
    a.ldx = ldx;
    a.y = y;
    a.ldy = ldy;
    a.plan = plan;
    a.acc0 = acc0;
    a.acc1 = acc1;
    a.done0 = ctrl;
    a.done1 = ctrl + sh.S;
    a.gen = ctrl + 2 * sh.S;
    a.exits = a.gen + 1;
    a.err = err;
    a.T = T;
    a.xdiv = xdiv;
    a.S = sh.S;
    a.n = sh.n;
    a.k = sh.k;
    a.r_max = sh.r_max;
    for (int i = 0; i <= LORA_MAX_SLICES; ++i) a.off[i] = sh.off[i];
    e = cudaFuncSetAttribute(tma_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tma_decode_kernel, a);
}

}  // namespace lora
