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
//   * One CTA per SM, about 110 KB of shared memory, so that the CTA of the
//     next call (launched as a programmatic dependent) fits beside it.  The
//     next call's producer warp issues its first stages of adapter weights
//     before griddepcontrol.wait: the weights never depend on the previous
//     layer, so their first burst overlaps the previous call's tail.  Only x,
//     y and the workspace wait for the previous grid.
//   * Stages of up to 32 KB in a ring of three, one mbarrier each.  A shrink
//     stage holds, for one slot, one group of its tokens and a run of 64-column
//     k-blocks, every slice's A rows (TMA 2D boxes of [r][64] bf16, 128-byte
//     swizzle, one per slice and k-block) and the group's x rows (16-byte
//     cp.async copies, gathered through sorted_ids by a second warp into the
//     same swizzled layout).  An expand stage holds a [64 columns][64 ranks]
//     box of B (ranks past r are the tensor map's zero fill) and the group's y
//     rows of those 64 columns.
//   * Four warps run mma.m16n8k16 (bf16, fp32 accumulate) from the staged
//     tiles with ldmatrix.  The shrink keeps its sums in registers across the
//     k-blocks of a run and adds them into an fp32 buffer (red.global.add.v2)
//     once per run; the split over k follows the byte-balanced partition
//     (TensorRT-LLM LoRA serving page, "路径二:split-K 调优").  A per-slot
//     counter of finished k-blocks (release / acquire) tells the expand of
//     that slot, in the same kernel, that its sums are complete; the expand's
//     B tiles are already streaming meanwhile.
//   * The expand feeds the fp32 sums to its MMA rounded once to bf16 (2^-9
//     relative, what serving engines' expand kernels take), accumulates in
//     fp32 and writes y = bf16(y + s * acc), rounded once.
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

namespace lora {

// ---------------------------------------------------------------------------
// Slot table with tensor maps: the ordinary table (TableLayout), then a
// 128-byte block header {magic, S, n, k, slice offsets}, then for every slot
// s and slice i two CUtensorMaps of 128 bytes: A_s,i as [r][k] (box [r][64],
// 128-byte swizzle) and B_s,i as [d_i][r] (box [64][64], 128-byte swizzle,
// ranks past r zero-filled).
// ---------------------------------------------------------------------------
constexpr int32_t kTmaTableMagic = 0x4d414d54;

struct TmaTableLayout {
    size_t hdr, maps, bytes;
    __host__ __device__ TmaTableLayout(int32_t S, int32_t n) {
        hdr = (TableLayout(S, n).bytes + 127) & ~size_t(127);
        maps = hdr + 128;
        bytes = maps + size_t(S) * size_t(n) * 256;
    }
};

namespace {

constexpr int kThreads = 192;        // warp 0: TMA, warp 1: row gather, warps 2..5: MMA
constexpr int kMmaThreads = 128;
constexpr int kStages = 3;
constexpr int kStageBytes = 32768;
constexpr int kXaBytes = 64 * 72 * 2;  // expand sums of 64 tokens x (64 + 8) ranks, bf16
constexpr int kSmemBytes = kStages * kStageBytes + kXaBytes + 1024;  // + alignment slack
constexpr int kMaxGrid = 256;
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
    int32_t pad[4];
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
static_assert(sizeof(PlanHdr) + sizeof(CtaRec) * kMaxGrid == 128 + 256 * 32, "plan layout matches tma_plan_size");

__host__ __device__ inline int32_t cdiv(int32_t a, int32_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int32_t pad16i(int32_t v) { return (v + 15) & ~15; }

struct TArgs {
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    const unsigned char *plan;
    float *acc0, *acc1;        // [n][T][r_max] fp32 sums, set g & 1 this call
    int32_t *done0, *done1;    // [S] finished k-blocks per slot
    int32_t *gen, *exits;      // call counter, CTAs that finished this call
    int32_t *err;
    int32_t T, S, n, k, r_max;
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
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, volatile int32_t *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kRingLimitNs) {
            *abort = 1;
            return false;
        }
    }
}

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

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, int32_t x, int32_t y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t &r0, uint32_t &r1, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// Not volatile: the data was published by an mbarrier wait (a volatile asm
// with a memory clobber) that precedes every use, so the compiler may hoist
// these loads ahead of the stores that follow them.
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_v2(float *p, float a, float b) {
    asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1,%2};" :: "l"(p), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ float2 ldcg_f2(const float *p) {
    float2 v;
    asm volatile("ld.global.cg.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ void stg32(void *p, uint32_t v) {
    asm volatile("st.global.b32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void mma_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Byte offset of 16-byte chunk `ch` of row `row` in a tile of 128-byte rows
// with the 128-byte swizzle (chunk index XOR row mod 8; tile 1024-aligned).
__device__ __forceinline__ uint32_t swz(int row, int ch) {
    return static_cast<uint32_t>(row) * 128u + (static_cast<uint32_t>(ch ^ (row & 7)) << 4);
}

// ---------------------------------------------------------------------------
// Walking a CTA's share of the plan
// ---------------------------------------------------------------------------
struct Slot {
    int32_t s, seg0, cnt, r, gs, ngs, cs, ge, nge;
    float scale;
};

// The slot records a CTA touches sit in a window of kSlotCache consecutive
// tiles from its first one (both of its lists are in slot order); the window
// is copied to shared memory in the prologue and tiles past it read the plan.
constexpr int kSlotCache = 32;

__device__ __forceinline__ Slot load_slot(const unsigned char *plan, int32_t a, const int4 *cache, int32_t base) {
    int4 v0, v1, v2;
    if (a >= base && a < base + kSlotCache) {
        const int4 *p = cache + 4 * (a - base);
        v0 = p[0];
        v1 = p[1];
        v2 = p[2];
    } else {
        const int4 *p = reinterpret_cast<const int4 *>(plan + plan_slots_off() + size_t(a) * sizeof(SlotRec));
        v0 = __ldcg(p);
        v1 = __ldcg(p + 1);
        v2 = __ldcg(p + 2);
    }
    Slot s;
    s.s = v0.x;
    s.seg0 = v0.y;
    s.cnt = v0.z;
    s.r = v0.w;
    s.scale = __int_as_float(v1.x);
    s.gs = v1.y;
    s.ngs = v1.z;
    s.cs = v1.w;
    s.ge = v2.x;
    s.nge = v2.y;
    return s;
}

// A shrink stage: slot tile, token group g, k-blocks [kb, kb + nb); `first`
// and `last` mark the ends of a run (same tile and group).
struct SStage {
    int32_t g, kb, nb;
};

// An expand unit: token group g, slice i, 64-column block cb of the slice.
struct EUnit {
    int32_t g, i, cb;
};

struct Ctx {
    int32_t T, n, k, r_max, nkb, ublk;
    int32_t off[LORA_MAX_SLICES + 1];
    const unsigned char *plan;
    const int32_t *ids;
    const unsigned char *maps;
};

// Token ids of a group of up to 128 rows held by a warp: lane l keeps rows l,
// l + 32, l + 64 and l + 96; id_of must be called by all 32 lanes with a
// warp-uniform row >> 5.
__device__ __forceinline__ void load_ids(const int32_t *ids, int32_t gsz, int32_t lane, int32_t (&idq)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int32_t r = q * 32 + lane;
        idq[q] = r < gsz ? __ldcg(ids + r) : 0;
    }
}
__device__ __forceinline__ int32_t id_of(const int32_t (&idq)[4], int32_t row) {
    const int32_t q = row >> 5;
    const int32_t v = q == 0 ? idq[0] : (q == 1 ? idq[1] : (q == 2 ? idq[2] : idq[3]));
    return __shfl_sync(0xffffffffu, v, row & 31);
}

// Expand unit u (0 <= u < ublk) of a token group -> slice and column block.
__device__ __forceinline__ void unit_slice(const Ctx &C, int32_t u, int32_t &i, int32_t &cb) {
    i = 0;
    while (true) {
        const int32_t nb = cdiv(C.off[i + 1] - C.off[i], 64);
        if (u < nb || i + 1 >= C.n) break;
        u -= nb;
        ++i;
    }
    cb = u;
}

// ---------------------------------------------------------------------------
// MMA roles
// ---------------------------------------------------------------------------
// One shrink run (slot tile, token group g, run_len k-blocks): consumes its
// stages from the ring, keeps the sums in registers and adds them into the
// call's fp32 buffer at the end.  The M tiles (16 tokens) x N tiles (8 ranks)
// of the run are spread over the four warps as a WM x WN grid, WM the
// smallest of 1, 2, 4 that leaves each warp at most MTW M tiles: warp w takes
// M tiles w % WM + WM i and N tiles w / WM + WN j.
constexpr int kMTW = 2, kNTW = 12;

__device__ __forceinline__ void shrink_run(const Ctx &C, const Slot &sl, int32_t g, int32_t run_len, uint32_t &c,
                                           uint32_t ring, uint32_t bars, float *acc_buf, volatile int32_t *abort,
                                           int32_t mw, int32_t lane) {
    const int32_t nr = C.n * sl.r, ntt = nr >> 3;
    const int32_t gsz = min(sl.gs, sl.cnt - g * sl.gs), gpad = pad16i(gsz), mtc = gpad >> 4;
    const int32_t WM = mtc <= 2 ? 1 : (mtc <= 4 ? 2 : 4), WN = 4 / WM;
    const int32_t wm = mw % WM, wn = mw / WM;
    float acc[kMTW][kNTW][4];
#pragma unroll
    for (int im = 0; im < kMTW; ++im)
#pragma unroll
        for (int in = 0; in < kNTW; ++in)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[im][in][e] = 0.f;
    int32_t done_pieces = 0;
    while (done_pieces < run_len) {
        const int32_t nb = min(sl.cs, run_len - done_pieces);
        const uint32_t st = c % kStages;
        const bool ok = ring_wait(bars + 8 * st, (c / kStages) & 1, abort);
        if (ok) {
            const uint32_t sbase = ring + st * kStageBytes;
            const uint32_t xoff = static_cast<uint32_t>(nb * nr) * 128u;
            for (int32_t kbl = 0; kbl < nb; ++kbl) {
                const uint32_t abase = sbase + static_cast<uint32_t>(kbl * nr) * 128u;
                const uint32_t xbase = sbase + xoff + static_cast<uint32_t>(kbl * gpad) * 128u;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t af[kMTW][4];
#pragma unroll
                    for (int im = 0; im < kMTW; ++im) {
                        const int32_t mt = wm + WM * im;
                        if (mt < mtc) ldsm_x4(af[im], xbase + swz(mt * 16 + (lane & 15), 2 * ks + (lane >> 4)));
                    }
#pragma unroll
                    for (int in = 0; in < kNTW; ++in) {
                        const int32_t nt = wn + WN * in;
                        if (nt < ntt) {
                            uint32_t b0, b1;
                            ldsm_x2(b0, b1, abase + swz(nt * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1)));
#pragma unroll
                            for (int im = 0; im < kMTW; ++im)
                                if (wm + WM * im < mtc)
                                    mma_bf16_16816(acc[im][in], af[im][0], af[im][1], af[im][2], af[im][3], b0, b1);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (kStages + st));
        ++c;
        done_pieces += nb;
        if (!ok) return;
    }
    // sums of this run -> acc_buf[i][p][j]
    const int32_t gq = lane >> 2, q = lane & 3;
    const int32_t p0 = sl.seg0 + g * sl.gs;
#pragma unroll
    for (int im = 0; im < kMTW; ++im) {
        const int32_t mt = wm + WM * im;
        if (mt >= mtc) continue;
#pragma unroll
        for (int in = 0; in < kNTW; ++in) {
            const int32_t nt = wn + WN * in;
            if (nt >= ntt) continue;
            const int32_t col = nt * 8 + 2 * q;
            const int32_t i = col / sl.r, j = col - i * sl.r;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int32_t tok = mt * 16 + gq + 8 * h;
                if (tok < gsz)
                    red_v2(acc_buf + (static_cast<size_t>(i) * C.T + p0 + tok) * C.r_max + j, acc[im][in][2 * h],
                           acc[im][in][2 * h + 1]);
            }
        }
    }
}

// One expand unit from the ring: y rows of token group g (gsz tokens from
// sorted position p0), slice i, columns [cb * 64, cb * 64 + 64) of the slice;
// the sums are in the xa buffer (bf16, row stride xs elements).
__device__ __forceinline__ void expand_unit(const Ctx &C, const Slot &sl, const int32_t *rows, int32_t gsz,
                                            int32_t i, int32_t cb, uint32_t sbase, uint32_t xbuf, int32_t xs,
                                            uint16_t *y, int64_t ldy, int32_t mw, int32_t lane) {
    const int32_t mtc = pad16i(gsz) >> 4, ksteps = pad16i(sl.r) >> 4;
    const uint32_t bbase = sbase, ybase = sbase + 8192;
    float acc[4][2][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][t][e] = 0.f;
    for (int32_t ks = 0; ks < ksteps; ++ks) {
        uint32_t af[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
            if (mt < mtc)
                ldsm_x4(af[mt], xbuf + static_cast<uint32_t>((mt * 16 + (lane & 15)) * xs * 2) +
                                    static_cast<uint32_t>((2 * ks + (lane >> 4)) * 16));
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int32_t nt = 2 * mw + t;
            uint32_t b0, b1;
            ldsm_x2(b0, b1, bbase + swz(nt * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1)));
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
                if (mt < mtc) mma_bf16_16816(acc[mt][t], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
        }
    }
    const int32_t gq = lane >> 2, q = lane & 3;
    const int32_t di = C.off[i + 1] - C.off[i];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
        if (mt >= mtc) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int32_t tok = mt * 16 + gq + 8 * h;
            if (tok >= gsz) continue;
            const int64_t row = rows[tok];
            uint16_t *yrow = y + row * ldy + C.off[i] + cb * 64;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int32_t cl = (2 * mw + t) * 8 + 2 * q;
                if (cb * 64 + cl >= di) continue;
                const uint32_t yv = lds32(ybase + swz(tok, cl >> 3) + static_cast<uint32_t>((cl & 7) * 2));
                const float f0 = bf16lo_to_f32(yv) + sl.scale * acc[mt][t][2 * h];
                const float f1 = bf16hi_to_f32(yv) + sl.scale * acc[mt][t][2 * h + 1];
                stg32(yrow + cl, pack_bf16x2(f0, f1));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2) tma_decode_kernel(TArgs a) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kStages];  // full[kStages], then empty[kStages]
    __shared__ int32_t s_abort, s_flag;
    __shared__ int32_t s_rows[kGe];                      // token ids of the expand run's group
    __shared__ int4 s_slots[4 * kSlotCache];              // slot records of tiles [slot_base, + kSlotCache)

    pdl_launch_dependents();
    const PlanHdr *H = reinterpret_cast<const PlanHdr *>(a.plan);
    const int4 h0 = __ldcg(reinterpret_cast<const int4 *>(H)), h1 = __ldcg(reinterpret_cast<const int4 *>(H) + 1);
    const int4 h2 = __ldcg(reinterpret_cast<const int4 *>(H) + 2), h3 = __ldcg(reinterpret_cast<const int4 *>(H) + 3);
    const uint64_t table = __ldcg(&H->table);
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
    const CtaRec *cr = reinterpret_cast<const CtaRec *>(a.plan + plan_ctas_off(a.S)) + blockIdx.x;
    const int4 crs = __ldcg(reinterpret_cast<const int4 *>(cr)), cre = __ldcg(reinterpret_cast<const int4 *>(cr) + 1);
    const int32_t slot_base = min(crs.x, cre.x);
    {
        const int32_t na = h1.z;
        const int32_t e = threadIdx.x;  // 128 int4: four per cached record
        if (e < 4 * kSlotCache && slot_base + (e >> 2) < na)
            s_slots[e] = __ldcg(reinterpret_cast<const int4 *>(a.plan + plan_slots_off() +
                                                                size_t(slot_base) * sizeof(SlotRec)) + e);
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(bar0 + 8 * st, 1 + 32);         // producer's expect_tx + 32 gather lanes
            mbar_init(bar0 + 8 * (kStages + st), 4);  // one arrival per MMA warp
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_abort = 0;
    }
    __syncthreads();

    const int32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
                const int32_t kb = idx % C.nkb;
                const int32_t nb = min(min(sl.cs, C.nkb - kb), left);
                const uint32_t st = c % kStages;
                if (c >= kStages && !ring_wait(bar0 + 8 * (kStages + st), ((c / kStages) + 1) & 1, abort)) break;
                const uint32_t full = bar0 + 8 * st, dst = ring + st * kStageBytes;
                mbar_expect_tx(full, static_cast<uint32_t>(nb * C.n * sl.r) * 128u);
                for (int32_t kbl = 0; kbl < nb; ++kbl)
                    for (int32_t i = 0; i < C.n; ++i)
                        tma_load_2d(dst + static_cast<uint32_t>((kbl * C.n + i) * sl.r) * 128u,
                                    C.maps + (static_cast<size_t>(sl.s) * C.n + i) * 256, (kb + kbl) * 64, 0, full,
                                    policy);
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
                const uint32_t st = c % kStages;
                if (c >= kStages && !ring_wait(bar0 + 8 * (kStages + st), ((c / kStages) + 1) & 1, abort)) break;
                const uint32_t full = bar0 + 8 * st;
                mbar_expect_tx(full, 8192u);
                tma_load_2d(ring + st * kStageBytes, C.maps + (static_cast<size_t>(sl.s) * C.n + i) * 256 + 128, 0,
                            cb * 64, full, policy);
                ++c;
                ++idx;
                --left;
                if (idx == sl.nge * C.ublk) {
                    ++tile;
                    idx = 0;
                }
            }
        }
    } else if (warp == 1) {
        // ---- row gather: x rows of shrink stages, y rows of expand units.  The
        // ids of the current token group stay in registers (lane l: rows l + 32 q),
        // so a stage issues its copies without waiting on any global load.
        pdl_wait();
        uint32_t c = 0;
        int32_t tile = crs.x, idx = crs.y, left = crs.z, cur = -1, cur_g = -1;
        int32_t idq[4] = {0, 0, 0, 0};
        Slot sl{};
        while (left > 0 && !*abort) {
            if (tile != cur) {
                sl = load_slot(C.plan, tile, s_slots, slot_base);
                cur = tile;
                cur_g = -1;
            }
            const int32_t g = idx / C.nkb, kb = idx % C.nkb;
            const int32_t nb = min(min(sl.cs, C.nkb - kb), left);
            const int32_t gsz = min(sl.gs, sl.cnt - g * sl.gs), gpad = pad16i(gsz);
            if (g != cur_g) {
                load_ids(C.ids + sl.seg0 + g * sl.gs, gsz, lane, idq);
                cur_g = g;
            }
            const uint32_t st = c % kStages;
            if (c >= kStages && !ring_wait(bar0 + 8 * (kStages + st), ((c / kStages) + 1) & 1, abort)) break;
            const uint32_t xdst = ring + st * kStageBytes + static_cast<uint32_t>(nb * C.n * sl.r) * 128u;
            const int32_t per_kb = gpad * 8;  // a multiple of 128: a warp's 32 elements share kbl and row >> 5
            for (int32_t e0 = 0; e0 < nb * per_kb; e0 += 32) {
                const int32_t e = e0 + lane;
                const int32_t kbl = e / per_kb, rem = e - kbl * per_kb, row = rem >> 3, ch = rem & 7;
                const int64_t tok = id_of(idq, row);
                cp16(xdst + static_cast<uint32_t>(kbl * gpad) * 128u + swz(row, ch),
                     a.x + tok * a.ldx + (kb + kbl) * 64 + ch * 8, row < gsz);
            }
            cp_arrive_noinc(bar0 + 8 * st);
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
        while (left > 0 && !*abort) {
            if (tile != cur) {
                sl = load_slot(C.plan, tile, s_slots, slot_base);
                cur = tile;
                cur_g = -1;
            }
            const int32_t g = idx / C.ublk;
            int32_t i, cb;
            unit_slice(C, idx % C.ublk, i, cb);
            const int32_t gsz = min(sl.ge, sl.cnt - g * sl.ge), gpad = pad16i(gsz);
            if (g != cur_g) {
                load_ids(C.ids + sl.seg0 + g * sl.ge, gsz, lane, idq);
                cur_g = g;
            }
            const int32_t di = C.off[i + 1] - C.off[i];
            const uint32_t st = c % kStages;
            if (c >= kStages && !ring_wait(bar0 + 8 * (kStages + st), ((c / kStages) + 1) & 1, abort)) break;
            const uint32_t ydst = ring + st * kStageBytes + 8192u;
            for (int32_t e0 = 0; e0 < gpad * 8; e0 += 32) {
                const int32_t e = e0 + lane;
                const int32_t row = e >> 3, ch = e & 7;
                const int32_t col = cb * 64 + ch * 8;
                const bool v = row < gsz && col < di;
                const int64_t tok = id_of(idq, row);
                cp16(ydst + swz(row, ch), a.y + tok * a.ldy + C.off[i] + (v ? col : 0), v);
            }
            cp_arrive_noinc(bar0 + 8 * st);
            ++c;
            ++idx;
            --left;
            if (idx == sl.nge * C.ublk) {
                ++tile;
                idx = 0;
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // ---- MMA warps
        pdl_wait();
        const int32_t mw = warp - 2, mtid = threadIdx.x - 64;
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
        uint32_t c = 0;
        int32_t tile = crs.x, idx = crs.y, left = crs.z;
        while (left > 0 && !*abort) {
            const Slot sl = load_slot(C.plan, tile, s_slots, slot_base);
            const int32_t g = idx / C.nkb, kb = idx % C.nkb;
            const int32_t run_len = min(C.nkb - kb, left);
            shrink_run(C, sl, g, run_len, c, ring, bar0, acc_buf, abort, mw, lane);
            mma_barrier();  // every warp's sums of the run are issued
            if (mtid == 0) {
                __threadfence();
                atomicAdd(done + sl.s, run_len);
            }
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
        while (left > 0 && !*abort) {
            const Slot sl = load_slot(C.plan, tile, s_slots, slot_base);
            const int32_t g = idx / C.ublk;
            int32_t i, cb;
            unit_slice(C, idx % C.ublk, i, cb);
            const int32_t blocks_i = cdiv(C.off[i + 1] - C.off[i], 64);
            const int32_t run_len = min(blocks_i - cb, left);
            const int32_t gsz = min(sl.ge, sl.cnt - g * sl.ge), gpad = pad16i(gsz);
            const int32_t p0 = sl.seg0 + g * sl.ge;
            const int32_t r16 = pad16i(sl.r), xs = r16 + 8;
            // the slot's sums are complete once every k-block of every group is in
            if (mtid == 0) {
                const int32_t need = sl.ngs * C.nkb;
                int32_t ok = 1;
                if (ld_acquire(done + sl.s) < need) {
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
            const bool ok = s_flag != 0;
            if (ok) {
                // the group's sums -> bf16 in the xa buffer; every load of a thread is
                // issued before its first store (at most 64 rows x 32 pairs / 128 threads)
                if (mtid < gsz) s_rows[mtid] = __ldcg(C.ids + p0 + mtid);
                const int32_t pairs = r16 >> 1, total = gpad * pairs;
                constexpr int kPer = kGe * 32 / kMmaThreads;
                float2 v[kPer];
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int32_t e = mtid + u * kMmaThreads;
                    const int32_t row = e / pairs, j = 2 * (e - row * pairs);
                    v[u] = make_float2(0.f, 0.f);
                    if (e < total && row < gsz && j < sl.r)
                        v[u] = ldcg_f2(acc_buf + (static_cast<size_t>(i) * C.T + p0 + row) * C.r_max + j);
                }
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int32_t e = mtid + u * kMmaThreads;
                    const int32_t row = e / pairs, j = 2 * (e - row * pairs);
                    if (e < total) sts32(xbuf + static_cast<uint32_t>((row * xs + j) * 2), pack_bf16x2(v[u].x, v[u].y));
                }
            }
            mma_barrier();
            for (int32_t u = 0; u < run_len; ++u) {
                const uint32_t st = c % kStages;
                const bool got = ring_wait(bar0 + 8 * st, (c / kStages) & 1, abort);
                if (got && ok)
                    expand_unit(C, sl, s_rows, gsz, i, cb + u, ring + st * kStageBytes, xbuf, xs, a.y, a.ldy, mw,
                                lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar0 + 8 * (kStages + st));
                ++c;
                if (!got) break;
            }
            mma_barrier();  // the xa buffer is read by every warp before the next run rewrites it
            idx += run_len;
            left -= run_len;
            if (idx == sl.nge * C.ublk) {
                ++tile;
                idx = 0;
            }
        }
    }

    __syncthreads();
    if (threadIdx.x == 0) {
        if (*abort) {
            report_error(a.err, LORA_ERR_TIMEOUT);
            // copies a stalled ring may still have in flight land within microseconds
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
        }
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
    const int32_t n = sh.n, nkb = sh.k / 64;
    int32_t ublk = 0;
    for (int i = 0; i < n; ++i) ublk += cdiv(sh.off[i + 1] - sh.off[i], 64);
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
        const int32_t cs = max(1, min(nkb, 256 / (nr + pad16i(gs))));
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
        rec.wps = (nr + gs) * 8;          // A rows and x rows of one k-block, 16-byte units
        rec.wpe = 8 * r + 16 * ge;        // B tile [64][r] and y rows read + written
        for (int q = 0; q < 4; ++q) rec.pad[q] = 0;
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
    for (int32_t s = 0; s < sh.S; ++s) {
        const int32_t r = ranks[s];
        if (r <= 0 || r > 256) continue;
        for (int32_t i = 0; i < sh.n; ++i) {
            CUtensorMap *ma = reinterpret_cast<CUtensorMap *>(p + L.maps + (size_t(s) * sh.n + i) * 256);
            const cuuint64_t adim[2] = {static_cast<cuuint64_t>(sh.k), static_cast<cuuint64_t>(r)};
            const cuuint64_t astr[1] = {static_cast<cuuint64_t>(sh.k) * 2};
            const cuuint32_t abox[2] = {64, static_cast<cuuint32_t>(r)};
            const cuuint32_t one[2] = {1, 1};
            if (enc(ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, reinterpret_cast<void *>(A_ptrs[s * sh.n + i]), adim,
                    astr, abox, one, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return false;
            CUtensorMap *mb = ma + 1;
            const int32_t di = sh.off[i + 1] - sh.off[i];
            const cuuint64_t bdim[2] = {static_cast<cuuint64_t>(r), static_cast<cuuint64_t>(di)};
            const cuuint64_t bstr[1] = {static_cast<cuuint64_t>(r) * 2};
            const cuuint32_t bbox[2] = {64, 64};
            if (enc(mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, reinterpret_cast<void *>(B_ptrs[s * sh.n + i]), bdim,
                    bstr, bbox, one, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
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
    int num_sms = 0;
    cudaError_t e = static_cast<cudaError_t>(num_sms_now(num_sms));
    if (e != cudaSuccess) return e;
    if (num_sms > kMaxGrid) return cudaErrorNotSupported;
    PArgs pa{sorted_ids, seg, active, err, T, num_sms};
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
// the two fp32 sum sets of [n][T][r_max].
cudaError_t launch_tma_decode(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                              const unsigned char *plan, float *acc0, float *acc1, int32_t *ctrl, int32_t T,
                              int32_t *err, cudaStream_t stream) {
    if (!decode_tma_supported(T, sh)) return cudaErrorNotSupported;
    int num_sms = 0;
    cudaError_t e = static_cast<cudaError_t>(num_sms_now(num_sms));
    if (e != cudaSuccess) return e;
    if (num_sms > kMaxGrid) return cudaErrorNotSupported;
    TArgs a;
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
    a.S = sh.S;
    a.n = sh.n;
    a.k = sh.k;
    a.r_max = sh.r_max;
    for (int i = 0; i <= LORA_MAX_SLICES; ++i) a.off[i] = sh.off[i];
    e = cudaFuncSetAttribute(tma_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms));
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
