// Decode-size LoRA branch as two kernels in which every warp is its own
// streaming engine (LORA_PATH_DECODE_DIRECT).
//
// At decode the branch reads each active adapter's A and B once while x and y
// are small (llama.cpp LoRA adapter page, section "为什么低秩增量可以「后加」":
// the low-rank branch is bandwidth-bound at decode), so the kernels are built
// to keep many bytes in flight on every SM with as little per-byte work as
// possible:
//
//   * Lane-private staging.  Each warp owns a ring of stages in shared memory.
//     A stage is a list of 512-byte chunks; lane l copies 16 bytes into bytes
//     [16 l, 16 l + 16) of a chunk (cp.async, zero-filled where a row or column
//     is out of range) and later reads back exactly those bytes as one of its
//     MMA fragments.  No lane ever reads another lane's bytes, so a stage needs
//     no barrier, no mbarrier and no ldmatrix: cp.async.wait_group is the only
//     synchronisation, and the warps of a CTA never wait for one another.
//   * Fragment order instead of data order.  mma.m16n8k16 sums over k, so any
//     fixed permutation of k that both operands share is allowed: lane 4g + q
//     reads the 16 contiguous bytes at columns 8q..8q+7 of a 32-column block of
//     its row and feeds columns 8q..8q+3 to the first k16 MMA, 8q+4..8q+7 to the
//     second.  Rows are permuted the same way, so that a lane's accumulators
//     cover 2 or 4 adjacent ranks (shrink: one red.v2/red.v4 per token) or 8
//     adjacent output columns (expand: one 16-byte load and store of y).
//   * Byte-balanced split.  The work is a list of units (shrink: slot, slice,
//     32-rank block, 32-column blocks of k; expand: slot, slice, 64 output
//     columns, 16 tokens) with a weight of about the HBM bytes they move; warp
//     w of W takes the pieces whose weight offset lies in its W-th of the
//     total, so big slots are split over k across many warps (split-K,
//     TensorRT-LLM LoRA serving page, "路径二:split-K 调优") and every warp of
//     the GPU moves about the same bytes.
//   * Shrink partial sums go to an fp32 buffer with vector reductions
//     (red.global.add.v4.f32).  The expand is launched as a programmatic
//     dependent of the shrink: it builds its tables and copies its first
//     stages of B and y (which the shrink does not write) before
//     griddepcontrol.wait, and reads the sums only after it.  The fp32 sums
//     enter the expand MMA rounded once to bf16 (2^-9 relative, as serving
//     engines feed their expand), accumulation stays fp32, and
//     y = bf16(y + s · xa B^T) is rounded once.
//   * The workspace holds two sum buffers and a call counter g: call g adds
//     into buffer g & 1 and clears buffer (g + 1) & 1, which the previous call
//     used; the last expand CTA to finish advances g.  No CTA waits on another.
//
//   * FP8 adapters (LORA_PATH_DECODE_DIRECT_FP8; TensorRT-LLM LoRA serving
//     page, "第五步:FP8 特判"): A and B are float8_e4m3fn codes.  The shrink
//     copies 64-column blocks (a lane's 16 bytes of A are 16 columns), converts
//     its x columns from bf16 to e4m3 in registers (clamped to +-448, nearest
//     even) and runs mma.m16n8k32 e4m3 with the same shared k-permutation;
//     token groups are 24 so that a block's 2 MT + 6 chunks fit a stage.  The
//     expand copies [64][r] bytes of B, converts them exactly to bf16 and feeds
//     a bf16 MMA with the sums split into bf16 hi and lo parts (about 2^-17 of
//     each sum, with fp32's exponent range).
//
// Limits (the host routes other cases elsewhere): T <= 2048, r_max <= 64,
// S * n_slices <= 512, S <= 512; FP8 also k % 16 == 0.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace lora {

namespace {

constexpr int kSCtas = 2;            // shrink CTAs per SM
constexpr int kSWarps = 6;           // shrink warps per CTA (12 per SM, 3 per sub-partition)
constexpr int kECtas = 2;            // expand CTAs per SM
constexpr int kEWarps = 4;           // expand warps per CTA
constexpr int kChunk = 512;          // 16 bytes per lane
constexpr int kSChunks = 11;         // shrink stage: 11 chunks (5.5 KB)
constexpr int kSStages = 3;          // shrink ring depth per warp
constexpr int kEStages = 2;          // expand ring depth per warp
constexpr int kMaxTokens = 2048;
constexpr int kMaxRank = 64;
constexpr int kMaxSlots = 512;
constexpr int kMaxPtrs = 512;        // S * n_slices
constexpr int kRB = 32;              // shrink rank block
constexpr int kTGs = 32;             // shrink token group
constexpr int kCB = 64;              // expand output columns per unit
constexpr int kTGe = 16;             // expand token group

// Shrink and expand parameters of the bf16 (kF8 false) and e4m3 variants:
// shrink token group, x chunks per 8 tokens, columns of k per block; expand B
// chunks per 32 ranks.
template <bool kF8>
struct VP {
    static constexpr int32_t TG = kF8 ? 24 : kTGs;
    static constexpr int32_t XF = kF8 ? 2 : 1;
    static constexpr int32_t BC = kF8 ? 64 : 32;
    static constexpr int32_t BW = kF8 ? 4 : 8;
};

struct DArgs {
    const uint16_t *x;
    int64_t ldx;
    int32_t x_div;       // x row of sorted item p: p / x_div (routed experts sharing a token's row)
    uint16_t *y;
    int64_t ldy;
    const int32_t *sorted_ids;
    const int32_t *seg;
    const int32_t *active;
    float *acc0, *acc1;  // [n][T][r_max] fp32 sums: buffer g & 1 this call
    int32_t *gen;        // call counter g
    int32_t *exits;      // expand CTAs that finished this call
    int32_t *err;
    int32_t T;
    const unsigned char *plan;  // this kernel's table image from a plan, or null: build the tables
};

__host__ __device__ inline int32_t cdiv(int32_t a, int32_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sa(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// 16 bytes global -> shared through L2 only (A, x and y: nothing is re-read
// from L1), or 16 zero bytes when !valid (src is not read then).
__device__ __forceinline__ void cp16_cg(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void red_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1,%2,%3,%4};" :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}
__device__ __forceinline__ void red_v2(float *p, float a, float b) {
    asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1,%2};" :: "l"(p), "f"(a), "f"(b) : "memory");
}

__device__ __forceinline__ float4 ldg_f4(const float *p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// Bulk (TMA) copies of contiguous byte ranges (16-byte aligned, sizes
// multiples of 16), completion counted on an mbarrier.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
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
// Bounded wait on an mbarrier phase (a bulk copy of this warp): false after
// 200 ms, which only a broken memory system can cause.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        uint64_t t1;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
        if (t1 - t0 > 200ull * 1000 * 1000) return false;
    }
}

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// FP8 (float8_e4m3fn) operands
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint2 lds8(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
// Four bf16 values (two bf16x2 words, lowest column in the low half of lo) to
// four e4m3 codes, lowest column in byte 0: clamped to the finite range
// (+-448, satfinite) and rounded to nearest even, as x.clamp(-448, 448)
// .to(float8_e4m3fn) does; bf16 -> f32 is exact, so this rounds once.
__device__ __forceinline__ uint32_t e4m3x4_from_bf16x4(uint32_t lo, uint32_t hi) {
    uint32_t r;
    asm("{\n\t.reg .b16 l, h;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\t"
        "mov.b32 %0, {l, h};\n\t}"
        : "=r"(r)
        : "f"(bf16lo_to_f32(lo)), "f"(bf16hi_to_f32(lo)), "f"(bf16lo_to_f32(hi)), "f"(bf16hi_to_f32(hi)));
    return r;
}
// Two e4m3 codes (bits 0..15 of w; byte 0 -> low half) to f16x2, exactly:
// every e4m3 value, subnormals included, is a normal f16.
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t w) {
    uint32_t r;
    asm("{\n\t.reg .b16 c;\n\t"
        "cvt.u16.u32 c, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
        : "=r"(r) : "r"(w));
    return r;
}
// Two e4m3 codes (bits 0..15 of w; byte 0 -> low half) to bf16x2, exactly:
// every e4m3 value has at most 4 significant bits and an exponent in bf16's
// range, so the f16 values of the exact conversion above convert exactly too.
__device__ __forceinline__ uint32_t bf16x2_from_e4m3x2(uint32_t w) {
    const uint32_t h = f16x2_from_e4m3x2(w);
    float lo, hi;
    asm("{\n\t.reg .b16 l, u;\n\t"
        "mov.b32 {l, u}, %2;\n\t"
        "cvt.f32.f16 %0, l;\n\t"
        "cvt.f32.f16 %1, u;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(h));
    return pack_bf16x2(lo, hi);
}
// mma.m16n8k32 with e4m3 A and B, fp32 accumulate.  Lane 4g + q: a0 = (row g,
// k 4q..4q+3), a1 = (row g+8, k 4q..), a2 = (row g, k 4q+16..), a3 = (row g+8,
// k 4q+16..); b0 = (k 4q..4q+3, col g), b1 = (k 4q+16.., col g); the lowest k
// in the lowest byte.  Accumulators as for m16n8k16.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// ---------------------------------------------------------------------------
// Tables: one copy per CTA in shared memory, built by the prologue.
// ---------------------------------------------------------------------------
struct Tabs {
    int32_t *misc;     // [0] active count NA, [1] call counter, [3..5] table header; plans: [2] T,
                       // [6] variant, [18] k, [19] r_max (misc[18], misc[19] follow scb)
    int32_t *soff;     // [LORA_MAX_SLICES + 1] slice offsets
    int32_t *scb;      // [LORA_MAX_SLICES + 1] exclusive prefix of 64-column blocks per slice
    int32_t *tok;      // [T] sorted token ids (-1 where invalid)
    int32_t *act;      // [S + 1] active list as loaded
    int32_t *seg;      // [S + 2]
    int32_t *rank;     // [S]
    float *scale;      // [S]
    uint64_t *aptr;    // [S * n]
    uint64_t *bptr;    // [S * n]
    int32_t *a_slot;   // [S] per active slot: slot id
    int32_t *a_p0;     // [S] first sorted position
    int32_t *a_len;    // [S] tokens
    int32_t *a_r;      // [S] rank (0: no work)
    long long *a_pre;  // [S + 1] exclusive prefix of slot weights
};

constexpr int kMiscInts = 8 + 2 * (LORA_MAX_SLICES + 1) + 2;

__host__ __device__ inline size_t tabs_bytes(int32_t S, int32_t n, int32_t T) {
    size_t b = 4 * (kMiscInts + size_t(T) + (S + 1) + (S + 2) + 2 * size_t(S));
    b = (b + 15) & ~size_t(15);
    b += 16 * size_t(S) * n;                    // aptr, bptr
    b += 4 * 4 * size_t(S);                     // a_slot, a_p0, a_len, a_r
    b = (b + 15) & ~size_t(15);
    b += 8 * (size_t(S) + 1);                   // a_pre
    return (b + 15) & ~size_t(15);
}

__device__ Tabs carve(unsigned char *base, int32_t S, int32_t n, int32_t T) {
    Tabs t;
    int32_t *p = reinterpret_cast<int32_t *>(base);
    t.misc = p;
    t.soff = p + 8;
    t.scb = t.soff + LORA_MAX_SLICES + 1;
    t.tok = p + kMiscInts;
    t.act = t.tok + T;
    t.seg = t.act + S + 1;
    t.rank = t.seg + S + 2;
    t.scale = reinterpret_cast<float *>(t.rank + S);
    size_t off = 4 * (kMiscInts + size_t(T) + (S + 1) + (S + 2) + 2 * size_t(S));
    off = (off + 15) & ~size_t(15);
    t.aptr = reinterpret_cast<uint64_t *>(base + off);
    t.bptr = t.aptr + size_t(S) * n;
    t.a_slot = reinterpret_cast<int32_t *>(t.bptr + size_t(S) * n);
    t.a_p0 = t.a_slot + S;
    t.a_len = t.a_p0 + S;
    t.a_r = t.a_len + S;
    off += 16 * size_t(S) * n + 16 * size_t(S);
    off = (off + 15) & ~size_t(15);
    t.a_pre = reinterpret_cast<long long *>(base + off);
    return t;
}

// ---------------------------------------------------------------------------
// Unit weights: the 512-byte chunks a unit brings into the SM (what bounds a
// warp's time), the A rows re-read once per token group included.
// ---------------------------------------------------------------------------
// Shrink: rank block rb of a slot of rank r with L tokens, per 32-column block
// of k: 2 MT chunks of A rows per token group of 32, one chunk of x rows per 8
// tokens, and a fixed cost.
__device__ __forceinline__ int32_t s_mt(int32_t r, int32_t rb) { return r - kRB * rb > 16 ? 2 : 1; }
__device__ __forceinline__ int32_t s_block_w(int32_t r, int32_t L, int32_t rb, int32_t tg, int32_t xf) {
    return 2 * s_mt(r, rb) * cdiv(L, tg) + xf * cdiv(L, 8) + 1;
}
__device__ __forceinline__ long long s_slot_w(int32_t r, int32_t L, int32_t n, int32_t nkb, int32_t tg, int32_t xf) {
    long long w = 0;
    for (int32_t rb = 0; kRB * rb < r; ++rb) w += s_block_w(r, L, rb, tg, xf);
    return w * nkb * n;
}
// Expand: token group tg (16 tokens) of 64 output columns: bw chunks of B rows
// per 32 ranks (8 for bf16, 4 for e4m3), two chunks of y and 2 nkb chunks of
// sums per 8 tokens, and a fixed cost.
__device__ __forceinline__ int32_t e_unit_w(int32_t r, int32_t L, int32_t tg, int32_t bw) {
    const int32_t nt8 = min(2, cdiv(L - kTGe * tg, 8)), nkb = cdiv(r, 32);
    return bw * nkb + 2 * nt8 * (1 + nkb) + 2;
}
__device__ __forceinline__ int32_t e_cb_w(int32_t r, int32_t L, int32_t bw) {
    const int32_t nkb = cdiv(r, 32);
    return cdiv(L, kTGe) * (bw * nkb + 2) + 2 * cdiv(L, 8) * (1 + nkb);
}

__device__ __forceinline__ void cp4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(sa(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp8(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(sa(dst)), "l"(src) : "memory");
}

// Prologue: every table load of the CTA in flight at once, then the checks,
// the per-active-slot records and their weight prefix.  Ends with a barrier.
// Weight parameters (VP): for the shrink the token group (tg), the x chunks per
// 8 tokens (xf) and the columns of k per block (bc); for the expand tg is the B
// chunks per 32 ranks.
template <bool kExpand>
__device__ void build_tabs(const DArgs &a, const Shape &sh, const void *table, const Tabs &t, int32_t tg,
                           int32_t xf, int32_t bc) {
    const int32_t S = sh.S, n = sh.n, T = a.T;
    const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31;
    const TableView tab(table, S, n);
    const int32_t *hdr = static_cast<const int32_t *>(table);
    if (tid == 0) {
        cp4(t.misc + 3, hdr);
        cp4(t.misc + 4, hdr + 1);
        cp4(t.misc + 5, hdr + 2);
        if (a.gen != nullptr) cp4(t.misc + 1, a.gen);
        else t.misc[1] = 0;
        int32_t c = 0, o = 0;
#pragma unroll
        for (int i = 0; i <= LORA_MAX_SLICES; ++i) {
            if (i <= sh.n) o = sh.off[i];  // compile-time index: the shape stays in parameter space
            t.soff[i] = o;
            t.scb[i] = c;
            if (i < LORA_MAX_SLICES && i < sh.n) c += cdiv(sh.off[i + 1] - o, kCB);
        }
    }
    for (int i = tid; i < T; i += nthr) cp4(t.tok + i, a.sorted_ids + i);
    for (int s = tid; s <= S; s += nthr) cp4(t.act + s, a.active + s);
    for (int s = tid; s < S + 2; s += nthr) cp4(t.seg + s, a.seg + s);
    for (int s = tid; s < S; s += nthr) {
        cp4(t.rank + s, tab.rank + s);
        cp4(t.scale + s, tab.scale + s);
    }
    for (int e = tid; e < S * n; e += nthr) {
        cp8(t.aptr + e, tab.a_ptr + e);
        cp8(t.bptr + e, tab.b_ptr + e);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    for (int i = tid; i < T; i += nthr) {
        const int32_t v = t.tok[i];
        if (v < 0 || v >= T) {
            if (blockIdx.x == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
            t.tok[i] = -1;
        }
    }
    const bool ok = t.misc[3] == kTableMagic && t.misc[4] == S && t.misc[5] == n && t.seg[S + 1] == T;
    if (!ok && tid == 0 && blockIdx.x == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
    const int32_t NA = ok ? min(max(t.act[0], 0), S) : 0;
    const int32_t nkb = cdiv(sh.k, bc), ncb = t.scb[LORA_MAX_SLICES];
    for (int j = tid; j < NA; j += nthr) {
        const int32_t s = t.act[1 + j];
        int32_t r = 0, L = 0, p0 = 0;
        if (s >= 0 && s < S) {
            p0 = t.seg[s];
            L = t.seg[s + 1] - p0;
            r = t.rank[s];
            if (p0 < 0 || L < 0 || p0 + L > T) {
                if (blockIdx.x == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
                r = 0;
            }
            if (r > sh.r_max || r > kMaxRank) {
                if (blockIdx.x == 0) report_error(a.err, LORA_ERR_RANK);
                r = 0;
            }
        } else if (blockIdx.x == 0) {
            report_error(a.err, LORA_ERR_INVALID_ARG);
        }
        if (r <= 0 || L <= 0) r = L = 0;
        t.a_slot[j] = max(s, 0);
        t.a_p0[j] = p0;
        t.a_len[j] = L;
        t.a_r[j] = r;
        t.a_pre[j] = r == 0 ? 0 : (kExpand ? static_cast<long long>(ncb) * e_cb_w(r, L, tg) : s_slot_w(r, L, n, nkb, tg, xf));
    }
    __syncthreads();
    if (warp == 0) {
        long long carry = 0;
        for (int32_t base = 0; base < NA; base += 32) {
            const int32_t j = base + lane;
            const long long v = j < NA ? t.a_pre[j] : 0;
            long long incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long w = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += w;
            }
            if (j < NA) t.a_pre[j] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            t.a_pre[NA] = carry;
            t.misc[0] = NA;
        }
    }
    __syncthreads();
}

// Prologue from a plan: the table image a plan kernel built with build_tabs
// for this shape and batch, copied in 16-byte pieces, then the call counter
// read fresh.  An image for another batch size or table is reported and leaves
// the call without work.  Ends with a barrier.
template <bool kF8>
__device__ void load_plan(const DArgs &a, const Shape &sh, const Tabs &t, size_t bytes) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    unsigned char *dst = reinterpret_cast<unsigned char *>(t.misc);
    for (size_t o = 16 * static_cast<size_t>(tid); o < bytes; o += 16 * static_cast<size_t>(nthr))
        cp16_cg(sa(dst + o), a.plan + o, true);
    cp_commit();
    cp_wait<0>();
    __syncthreads();
    if (tid == 0) {
        t.misc[1] = *reinterpret_cast<volatile const int32_t *>(a.gen);
        // everything that sets an address must match: batch, counts, variant, k, r_max, slice offsets
        bool ok = t.misc[2] == a.T && t.misc[3] == kTableMagic && t.misc[4] == sh.S && t.misc[5] == sh.n &&
                  t.misc[6] == (kF8 ? 1 : 0) && t.misc[18] == sh.k && t.misc[19] == sh.r_max;
#pragma unroll
        for (int i = 0; i <= LORA_MAX_SLICES; ++i)
            if (i <= sh.n && t.soff[i] != sh.off[i]) ok = false;  // compile-time index into the shape
        if (!ok) {
            if (blockIdx.x == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
            t.misc[0] = 0;
            t.a_pre[0] = 0;
        }
    }
    __syncthreads();
}

// Last active slot j in [0, NA) with a_pre[j] <= v.
__device__ __forceinline__ int32_t find_active(const long long *pre, int32_t NA, long long v) {
    int32_t lo = 0, hi = NA;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (pre[mid] <= v) lo = mid + 1;
        else hi = mid;
    }
    return lo - 1;
}

// This warp's share [R0, R1) of the total weight W.
template <int kWarpsPerCta>
__device__ __forceinline__ void warp_share(long long W, long long &R0, long long &R1) {
    const long long NW = static_cast<long long>(gridDim.x) * kWarpsPerCta;
    const long long gw = static_cast<long long>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
    R0 = (W * gw + NW - 1) / NW;
    R1 = (W * (gw + 1) + NW - 1) / NW;
}

// ---------------------------------------------------------------------------
// Shrink: xa[i][p][j] += sum over a block range of k of x[tok(p), c] A_{s,i}[j, c]
// ---------------------------------------------------------------------------
// A segment: the warp's blocks [bs, be) of unit (active slot ja, slice i,
// rank block rb) for token group g.  The warp walks its blocks of a unit once
// per token group; a segment's sums stay in registers and are reduced into the
// buffer after its last block.  Two walkers follow the same segments: the
// copy walker runs one stage ahead of the compute walker.
struct SGen {
    int32_t ja, i, rb, g, bs, be, w;
    long long start, R1;
    bool live;
};

__device__ __forceinline__ int32_t s_nt8(int32_t L, int32_t g, int32_t tg) { return min(tg / 8, cdiv(L - tg * g, 8)); }

// Blocks of the current unit whose weight start is below R1.
__device__ __forceinline__ void s_range(SGen &c, int32_t nkb) {
    const long long lim = c.R1 - c.start;
    c.be = lim <= 0 ? 0 : static_cast<int32_t>(min(static_cast<long long>(nkb), (lim + c.w - 1) / c.w));
    c.g = 0;
    if (c.be <= c.bs) c.live = false;
}

template <bool kF8>
__device__ __forceinline__ void s_next_unit(SGen &c, const Tabs &t, int32_t n, int32_t nkb) {
    c.start += static_cast<long long>(nkb) * c.w;
    if (kRB * (++c.rb) >= t.a_r[c.ja]) {
        c.rb = 0;
        if (++c.i == n) {
            c.i = 0;
            const int32_t NA = t.misc[0];
            do {
                ++c.ja;
            } while (c.ja < NA && t.a_r[c.ja] == 0);
            if (c.ja >= NA) {
                c.live = false;
                return;
            }
        }
    }
    c.w = s_block_w(t.a_r[c.ja], t.a_len[c.ja], c.rb, VP<kF8>::TG, VP<kF8>::XF);
    c.bs = 0;
    s_range(c, nkb);
}

template <bool kF8>
__device__ __forceinline__ void s_next_seg(SGen &c, const Tabs &t, int32_t n, int32_t nkb) {
    if (VP<kF8>::TG * (++c.g) >= t.a_len[c.ja]) s_next_unit<kF8>(c, t, n, nkb);
}

template <bool kF8>
__device__ __forceinline__ void s_first(SGen &c, const Tabs &t, int32_t n, int32_t nkb) {
    const int32_t NA = t.misc[0];
    c.ja = c.i = c.rb = c.g = c.bs = c.be = 0;  // defined fields for a warp without work
    c.w = 1;
    c.start = 0;
    long long R0;
    warp_share<kSWarps>(t.a_pre[NA], R0, c.R1);
    c.live = R0 < c.R1;
    if (!c.live) return;
    c.ja = find_active(t.a_pre, NA, R0);
    const int32_t r = t.a_r[c.ja], L = t.a_len[c.ja];
    long long o = R0 - t.a_pre[c.ja];
    constexpr int32_t tg = VP<kF8>::TG, xf = VP<kF8>::XF;
    const long long wslice = s_slot_w(r, L, 1, nkb, tg, xf);
    c.i = static_cast<int32_t>(o / wslice);
    o -= c.i * wslice;
    c.start = t.a_pre[c.ja] + c.i * wslice;
    c.rb = 0;
    while (true) {
        const long long wu = static_cast<long long>(nkb) * s_block_w(r, L, c.rb, tg, xf);
        if (o < wu) break;
        o -= wu;
        c.start += wu;
        ++c.rb;
    }
    c.w = s_block_w(r, L, c.rb, tg, xf);
    c.bs = static_cast<int32_t>((o + c.w - 1) / c.w);
    if (c.bs >= nkb) {
        s_next_unit<kF8>(c, t, n, nkb);  // the share starts after this unit's last block start
        return;
    }
    s_range(c, nkb);
}

// Copy walker: per-segment lane pointers at block 0, so a block costs one
// 64-bit add per 16-byte copy.  Chunk c < 2 MT of a block is A row
// 2 MT gq + c of the rank block; chunk 2 MT + nt is the x row of token
// tg g + 8 nt + gq; lane 4 gq + q copies columns 8q..8q+7 of each.  With FP8
// weights (kF8) a block is 64 columns: the lane's A chunk holds columns
// 16q..16q+15 (one byte each) and its x row, still bf16, takes the two chunks
// 2 MT + 2 nt and 2 MT + 2 nt + 1.
struct SCopy {
    SGen gen;
    int32_t b, kb, cpb, mt, nt;
    uint32_t vm;
    const unsigned char *pa[4], *px[4];
};

template <bool kF8>
__device__ __forceinline__ void s_copy_seg(SCopy &s, const Tabs &t, const Shape &sh, const DArgs &a, int lane) {
    constexpr int32_t kEB = kF8 ? 1 : 2;  // bytes per weight
    const int32_t gq = lane >> 2, q = lane & 3;
    constexpr int32_t tg = VP<kF8>::TG;
    const int32_t ja = s.gen.ja, r = t.a_r[ja], L = t.a_len[ja], p0 = t.a_p0[ja];
    s.mt = s_mt(r, s.gen.rb);
    s.nt = s_nt8(L, s.gen.g, tg);
    s.cpb = 2 * s.mt + (kF8 ? 2 : 1) * s.nt;
    s.kb = kSChunks / s.cpb;
    s.b = s.gen.bs;
    const int32_t rows = min(kRB, r - kRB * s.gen.rb);
    const unsigned char *A = reinterpret_cast<const unsigned char *>(t.aptr[t.a_slot[ja] * sh.n + s.gen.i]) +
                             kEB * static_cast<int64_t>(kRB * s.gen.rb) * sh.k + 16 * q;
    uint32_t vm = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int32_t row = 2 * s.mt * gq + c;
        const bool v = c < 2 * s.mt && row < rows;
        s.pa[c] = A + (v ? kEB * static_cast<int64_t>(row) * sh.k : 0);
        vm |= v ? (1u << c) : 0u;
    }
    const unsigned char *X = reinterpret_cast<const unsigned char *>(a.x) + (kF8 ? 32 : 16) * q;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const int32_t jt = tg * s.gen.g + 8 * nt + gq;
        const int32_t tok = (nt < s.nt && jt < L) ? t.tok[p0 + jt] : -1;
        const int32_t xr = a.x_div == 1 ? tok : tok / a.x_div;
        s.px[nt] = X + (tok >= 0 ? 2 * static_cast<int64_t>(xr) * a.ldx : 0);
        vm |= tok >= 0 ? (1u << (4 + nt)) : 0u;
    }
    s.vm = vm;
}

// Issue the next stage of copies into `slot` (this lane's bytes) and commit
// a group (an empty one once the walk is over).
// kq = k minus the lane's first column in a block: a block's chunk is in range
// when (columns per block) * blk < kq.
template <bool kF8>
__device__ __forceinline__ void s_copy_stage(SCopy &s, uint32_t slot, int32_t kq, const Tabs &t, const Shape &sh,
                                             const DArgs &a, int lane, int32_t nkb) {
    if (s.gen.live) {
        const int32_t nb = min(s.kb, s.gen.be - s.b);
#pragma unroll(kF8 ? 1 : 4)
        for (int j = 0; j < 4; ++j) {
            if (j < nb) {
                const int32_t blk = s.b + j;
                const bool cv = (kF8 ? 64 : 32) * blk < kq;
                const uint32_t dst = slot + j * s.cpb * kChunk;
                const int64_t off = 64 * static_cast<int64_t>(blk);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (c < 2 * s.mt) cp16_cg(dst + c * kChunk, s.pa[c] + off, cv && ((s.vm >> c) & 1u));
                const uint32_t dx = dst + 2 * s.mt * kChunk;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    if (nt >= s.nt) continue;
                    const bool v = cv && ((s.vm >> (4 + nt)) & 1u);
                    if (kF8) {
                        cp16_cg(dx + 2 * nt * kChunk, s.px[nt] + 2 * off, v);
                        cp16_cg(dx + (2 * nt + 1) * kChunk, s.px[nt] + 2 * off + 16, v);
                    } else {
                        cp16_cg(dx + nt * kChunk, s.px[nt] + off, v);
                    }
                }
            }
        }
        s.b += nb;
        if (s.b >= s.gen.be) {
            s_next_seg<kF8>(s.gen, t, sh.n, nkb);
            if (s.gen.live) s_copy_seg<kF8>(s, t, sh, a, lane);
        }
    }
    cp_commit();
}

// Lane 4 gq + q holds, for tokens 8 nt + 2q + e, the ranks 2 MT gq .. + 2 MT - 1
// of the block: acc[mt][nt][e] is rank 2 MT gq + 2 mt, acc[mt][nt][2 + e] the next.
template <bool kF8>
__device__ __forceinline__ void s_reduce(const SGen &c, float *buf, const Tabs &t, const Shape &sh, int32_t T,
                                      int lane, const float (&acc)[2][4][4]) {
    const int32_t gq = lane >> 2, q = lane & 3;
    const int32_t r = t.a_r[c.ja], L = t.a_len[c.ja], p0 = t.a_p0[c.ja];
    constexpr int32_t tg = VP<kF8>::TG;
    const int32_t MT = s_mt(r, c.rb), NT8 = s_nt8(L, c.g, tg);
    const int32_t rows = min(kRB, r - kRB * c.rb);
    float *base = buf + (static_cast<int64_t>(c.i) * T + p0 + tg * c.g) * sh.r_max + kRB * c.rb;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        if (nt >= NT8) continue;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int32_t jt = 8 * nt + 2 * q + e;
            if (tg * c.g + jt >= L) continue;
            float *p = base + static_cast<int64_t>(jt) * sh.r_max;
            if (MT == 2) {
                if (4 * gq < rows) red_v4(p + 4 * gq, acc[0][nt][e], acc[0][nt][2 + e], acc[1][nt][e], acc[1][nt][2 + e]);
            } else {
                if (2 * gq < rows) red_v2(p + 2 * gq, acc[0][nt][e], acc[0][nt][2 + e]);
            }
        }
    }
}

size_t direct_shrink_smem(int32_t S, int32_t n, int32_t T) {
    return static_cast<size_t>(kSWarps) * kSStages * kSChunks * kChunk + tabs_bytes(S, n, T);
}

// kF8: A in e4m3, x converted to e4m3 in registers, 64-column blocks of k,
// token groups of 24 (a stage of 2 MT + 6 chunks holds one block).
template <bool kF8>
__global__ void __launch_bounds__(32 * kSWarps, kSCtas) direct_shrink_kernel(DArgs a, Shape sh, const void *table) {
    constexpr int32_t kTG = VP<kF8>::TG, kXF = VP<kF8>::XF, kBC = VP<kF8>::BC;
    extern __shared__ __align__(128) unsigned char smem[];
    // the expand may start its prologue as soon as every CTA of this grid runs
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Tabs t = carve(smem + static_cast<size_t>(kSWarps) * kSStages * kSChunks * kChunk, sh.S, sh.n, a.T);
    if (a.plan != nullptr) load_plan<kF8>(a, sh, t, tabs_bytes(sh.S, sh.n, a.T));
    else build_tabs<false>(a, sh, table, t, kTG, kXF, kBC);
    const int32_t gen = t.misc[1];
    float *buf = (gen & 1) ? a.acc1 : a.acc0;
    {
        // clear the buffer the previous call used: the next call adds into it
        float4 *other = reinterpret_cast<float4 *>((gen & 1) ? a.acc0 : a.acc1);
        const int64_t n4 = static_cast<int64_t>(sh.n) * a.T * sh.r_max / 4;
        for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid; e < n4;
             e += static_cast<int64_t>(gridDim.x) * blockDim.x)
            other[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int32_t nkb = cdiv(sh.k, kBC), kq = sh.k - (kBC / 4) * (lane & 3);
    const uint32_t ring = sa(smem) + warp * (kSStages * kSChunks * kChunk) + 16 * lane;
    constexpr uint32_t kSlot = kSChunks * kChunk;

    SCopy cw;
    s_first<kF8>(cw.gen, t, sh.n, nkb);
    if (cw.gen.live) s_copy_seg<kF8>(cw, t, sh, a, lane);
    SGen cg = cw.gen;  // compute walker
#pragma unroll
    for (int s = 0; s < kSStages - 1; ++s) s_copy_stage<kF8>(cw, ring + s * kSlot, kq, t, sh, a, lane, nkb);

    float acc[2][4][4];
    int32_t sc = 0, si = kSStages - 1;
    int32_t b = cg.bs, kb = 1, cpb = 1, MT = 1, NT = 1;
    if (cg.live) {
        MT = s_mt(t.a_r[cg.ja], cg.rb);
        NT = s_nt8(t.a_len[cg.ja], cg.g, kTG);
        cpb = 2 * MT + kXF * NT;
        kb = kSChunks / cpb;
    }
    while (cg.live) {
        s_copy_stage<kF8>(cw, ring + si * kSlot, kq, t, sh, a, lane, nkb);
        si = si + 1 == kSStages ? 0 : si + 1;
        cp_wait<kSStages - 1>();
        if (b == cg.bs) {
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
        }
        const int32_t nb = min(kb, cg.be - b);
        const uint32_t slot = ring + sc * kSlot;
#pragma unroll(kF8 ? 1 : 4)
        for (int j = 0; j < 4; ++j) {
            if (j >= nb) continue;
            const uint32_t src = slot + j * cpb * kChunk;
            uint4 av[4], xv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) av[c] = c < 2 * MT ? lds16(src + c * kChunk) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                if (kF8) {
                    // columns 16q..16q+7 and 16q+8..16q+15 of the token's x row, to e4m3
                    const bool v = nt < NT;
                    const uint4 lo = v ? lds16(src + (2 * MT + 2 * nt) * kChunk) : make_uint4(0, 0, 0, 0);
                    const uint4 hi = v ? lds16(src + (2 * MT + 2 * nt + 1) * kChunk) : make_uint4(0, 0, 0, 0);
                    xv[nt] = make_uint4(e4m3x4_from_bf16x4(lo.x, lo.y), e4m3x4_from_bf16x4(lo.z, lo.w),
                                        e4m3x4_from_bf16x4(hi.x, hi.y), e4m3x4_from_bf16x4(hi.z, hi.w));
                } else {
                    xv[nt] = nt < NT ? lds16(src + (2 * MT + nt) * kChunk) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                if (mt >= MT) continue;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    if (nt >= NT) continue;
                    if (kF8) {
                        // columns 16q + 0..7 feed k {4q..4q+3, 4q+16..4q+19} of the first MMA, 16q + 8..15 the second
                        mma_e4m3_16832(acc[mt][nt], av[2 * mt].x, av[2 * mt + 1].x, av[2 * mt].y, av[2 * mt + 1].y,
                                       xv[nt].x, xv[nt].y);
                        mma_e4m3_16832(acc[mt][nt], av[2 * mt].z, av[2 * mt + 1].z, av[2 * mt].w, av[2 * mt + 1].w,
                                       xv[nt].z, xv[nt].w);
                    } else {
                        mma_bf16_16816(acc[mt][nt], av[2 * mt].x, av[2 * mt + 1].x, av[2 * mt].y, av[2 * mt + 1].y,
                                       xv[nt].x, xv[nt].y);
                        mma_bf16_16816(acc[mt][nt], av[2 * mt].z, av[2 * mt + 1].z, av[2 * mt].w, av[2 * mt + 1].w,
                                       xv[nt].z, xv[nt].w);
                    }
                }
            }
        }
        sc = sc + 1 == kSStages ? 0 : sc + 1;
        b += nb;
        if (b >= cg.be) {
            s_reduce<kF8>(cg, buf, t, sh, a.T, lane, acc);
            s_next_seg<kF8>(cg, t, sh.n, nkb);
            if (cg.live) {
                b = cg.bs;
                MT = s_mt(t.a_r[cg.ja], cg.rb);
                NT = s_nt8(t.a_len[cg.ja], cg.g, kTG);
                cpb = 2 * MT + kXF * NT;
                kb = kSChunks / cpb;
            }
        }
    }
    cp_wait<0>();
}

// ---------------------------------------------------------------------------
// Expand: y[tok(p), o_i + c] = bf16(y + s * sum_j xa[i][p][j] B_{s,i}[c, j])
// ---------------------------------------------------------------------------
// A unit: active slot ja, slice i, token group tg of 16, block ci of 64 output
// columns.  MMA rows are the
// 64 output columns (4 tiles of 16), MMA columns the tokens, k the rank.  One
// stage holds one unit: bytes [0, 8 KB) the unit's B rows 64 ci .. + 63 as
// stored ([64][r] bf16, one bulk copy, completion on the slot's mbarrier);
// then chunk c < 4 (lane-private cp.async) the y row of token
// 16 tg + 8 nt + 2q + e (c = 2 nt + e) at columns 64 ci + 8 gq...
// Lane 4 gq + q feeds MMA row m of tile mt from B row 8 (m % 8) + 2 mt + m / 8,
// so that its accumulators cover the 8 adjacent columns 8 gq .. 8 gq + 7.
constexpr uint32_t kEBTile = 8192;
constexpr uint32_t kESlot = kEBTile + 4 * kChunk;

struct EGen {
    int32_t ja, i, tg, ci;
    long long start, R1;
    bool live;
};

// Units of a slot in the order (slice, token group, column block): consecutive
// units of a warp mostly share their tokens' sums, which stay in registers.
template <bool kF8>
__device__ __forceinline__ void e_advance(EGen &c, const Tabs &t, int32_t n) {
    const int32_t r = t.a_r[c.ja], L = t.a_len[c.ja];
    c.start += e_unit_w(r, L, c.tg, VP<kF8>::BW);
    if (t.scb[c.i] + (++c.ci) == t.scb[c.i + 1]) {
        c.ci = 0;
        if (kTGe * (++c.tg) >= L) {
            c.tg = 0;
            if (++c.i == n) {
                c.i = 0;
                const int32_t NA = t.misc[0];
                do {
                    ++c.ja;
                } while (c.ja < NA && t.a_r[c.ja] == 0);
                if (c.ja >= NA) c.live = false;
            }
        }
    }
    if (c.start >= c.R1) c.live = false;
}

template <bool kF8>
__device__ __forceinline__ void e_first(EGen &c, const Tabs &t, int32_t n) {
    const int32_t NA = t.misc[0];
    c.ja = c.i = c.tg = c.ci = 0;  // defined fields for a warp without work
    c.start = 0;
    long long R0;
    warp_share<kEWarps>(t.a_pre[NA], R0, c.R1);
    c.live = R0 < c.R1;
    if (!c.live) return;
    c.ja = find_active(t.a_pre, NA, R0);
    const int32_t r = t.a_r[c.ja], L = t.a_len[c.ja];
    long long o = R0 - t.a_pre[c.ja];
    constexpr int32_t bw = VP<kF8>::BW;
    const long long wcb = e_cb_w(r, L, bw);
    c.start = t.a_pre[c.ja];
    while (o >= (t.scb[c.i + 1] - t.scb[c.i]) * wcb) {
        const long long ws = (t.scb[c.i + 1] - t.scb[c.i]) * wcb;
        o -= ws;
        c.start += ws;
        ++c.i;
    }
    const int32_t nci = t.scb[c.i + 1] - t.scb[c.i];
    while (true) {
        const long long wt = static_cast<long long>(nci) * e_unit_w(r, L, c.tg, bw);
        if (o < wt) break;
        o -= wt;
        c.start += wt;
        ++c.tg;
    }
    const int32_t w = e_unit_w(r, L, c.tg, bw);
    c.ci = static_cast<int32_t>(o / w);
    c.start += static_cast<long long>(c.ci) * w;
    // the first unit whose start is >= R0
    if (c.start < R0) e_advance<kF8>(c, t, n);
    if (c.start >= c.R1) c.live = false;
}

// Copies of the next unit into slot `slot` of this warp's ring (base `wslot`),
// then a commit (an empty group once the walk is over).  kF8: the B rows are
// e4m3, r bytes each.
template <bool kF8>
__device__ __forceinline__ void e_copy_stage(EGen &g, uint32_t wslot, uint32_t bar, const Tabs &t, const Shape &sh,
                                             const DArgs &a, int lane, int32_t n) {
    if (g.live) {
        const int32_t gq = lane >> 2, q = lane & 3;
        const int32_t ja = g.ja, r = t.a_r[ja], L = t.a_len[ja], p0 = t.a_p0[ja];
        const int32_t o0 = t.soff[g.i], d = t.soff[g.i + 1] - o0;
        if (lane == 0) {
            const int32_t rows = min(kCB, d - kCB * g.ci);
            constexpr int32_t kEB = kF8 ? 1 : 2;
            const uint32_t bytes = kEB * static_cast<uint32_t>(rows * r);
            const unsigned char *src = reinterpret_cast<const unsigned char *>(t.bptr[t.a_slot[ja] * sh.n + g.i]) +
                                       kEB * static_cast<int64_t>(kCB * g.ci) * r;
            mbar_expect_tx(bar, bytes);
            bulk_copy(wslot, src, bytes, bar);
        }
        const int32_t col0 = kCB * g.ci + 8 * gq;
        const unsigned char *Y = reinterpret_cast<const unsigned char *>(a.y) + 2 * static_cast<int64_t>(o0 + col0);
        const uint32_t ydst = wslot + kEBTile + 16 * lane;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            if (kTGe * g.tg + 8 * nt >= L) break;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int32_t jt = kTGe * g.tg + 8 * nt + 2 * q + e;
                const int32_t tok = jt < L ? t.tok[p0 + jt] : -1;
                const bool v = tok >= 0 && col0 < d;
                cp16_cg(ydst + (2 * nt + e) * kChunk, Y + (v ? 2 * static_cast<int64_t>(tok) * a.ldy : 0), v);
            }
        }
        e_advance<kF8>(g, t, n);
    }
    cp_commit();
}

// The sums of a unit's tokens 16 tg + 8 nt + gq at ranks 32 kb + 8q .. + 7.
__device__ __forceinline__ void e_load_xa(const EGen &g, const float *buf, const Tabs &t, const Shape &sh,
                                          int32_t T, int lane, float4 (&X)[2][2][2]) {
    const int32_t gq = lane >> 2, q = lane & 3;
    if (!g.live) {
        // past the warp's last unit: the tables are not indexed with its fields
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) X[nt][kb][0] = X[nt][kb][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int32_t ja = g.ja, r = t.a_r[ja], L = t.a_len[ja], p0 = t.a_p0[ja];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int32_t jt = kTGe * g.tg + 8 * nt + gq;
        const float *row = buf + (static_cast<int64_t>(g.i) * T + p0 + jt) * sh.r_max + 8 * q;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            const bool v = jt < L && 32 * kb + 8 * q < r;
            X[nt][kb][0] = v ? ldg_f4(row + 32 * kb) : make_float4(0.f, 0.f, 0.f, 0.f);
            X[nt][kb][1] = v ? ldg_f4(row + 32 * kb + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// kF8: B rows are e4m3 and enter a bf16 MMA (exact conversion); the sums
// enter it as two bf16 parts, hi = bf16(sum) and lo = bf16(sum - hi) (about
// 2^-17 of each sum, and no overflow: bf16 has fp32's exponent range), one
// MMA for each part.
template <bool kF8>
__device__ __forceinline__ void e_compute(const EGen &g, uint32_t wslot, const float4 (&X)[2][2][2], const Tabs &t,
                                          const DArgs &a, int lane) {
    const int32_t gq = lane >> 2, q = lane & 3;
    const int32_t ja = g.ja, r = t.a_r[ja], L = t.a_len[ja], p0 = t.a_p0[ja];
    const int32_t NT8 = min(2, cdiv(L - kTGe * g.tg, 8));
    float acc[4][2][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
        if (32 * kb >= r) break;
        uint32_t bh[2][2][2];  // [nt][half][pair]: the sums rounded to bf16 once (kF8: the hi part)
        uint32_t bl[2][2][2];  // kF8: the lo part
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (kF8) {
                    split_bf16x2(X[nt][kb][h].x, X[nt][kb][h].y, bh[nt][h][0], bl[nt][h][0]);
                    split_bf16x2(X[nt][kb][h].z, X[nt][kb][h].w, bh[nt][h][1], bl[nt][h][1]);
                } else {
                    bh[nt][h][0] = pack_bf16x2(X[nt][kb][h].x, X[nt][kb][h].y);
                    bh[nt][h][1] = pack_bf16x2(X[nt][kb][h].z, X[nt][kb][h].w);
                }
            }
        const int32_t rc = 32 * kb + 8 * q;
        const bool vk = rc < r;
        // B row 8 gq + 2 mt (+1) at ranks rc..rc+7: byte kEB (row r + rc) of the tile
        constexpr uint32_t kEB = kF8 ? 1u : 2u;
        const uint32_t brow = wslot + kEB * static_cast<uint32_t>(8 * gq * r + rc);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            uint4 c0, c1;
            if (kF8) {
                const uint2 v0 = vk ? lds8(brow + static_cast<uint32_t>(2 * mt * r)) : make_uint2(0, 0);
                const uint2 v1 = vk ? lds8(brow + static_cast<uint32_t>((2 * mt + 1) * r)) : make_uint2(0, 0);
                c0 = make_uint4(bf16x2_from_e4m3x2(v0.x), bf16x2_from_e4m3x2(v0.x >> 16), bf16x2_from_e4m3x2(v0.y),
                                bf16x2_from_e4m3x2(v0.y >> 16));
                c1 = make_uint4(bf16x2_from_e4m3x2(v1.x), bf16x2_from_e4m3x2(v1.x >> 16), bf16x2_from_e4m3x2(v1.y),
                                bf16x2_from_e4m3x2(v1.y >> 16));
            } else {
                c0 = vk ? lds16(brow + 2u * static_cast<uint32_t>(2 * mt * r)) : make_uint4(0, 0, 0, 0);
                c1 = vk ? lds16(brow + 2u * static_cast<uint32_t>((2 * mt + 1) * r)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                if (nt >= NT8) continue;
                if (kF8) {
                    mma_bf16_16816(acc[mt][nt], c0.x, c1.x, c0.y, c1.y, bh[nt][0][0], bh[nt][0][1]);
                    mma_bf16_16816(acc[mt][nt], c0.z, c1.z, c0.w, c1.w, bh[nt][1][0], bh[nt][1][1]);
                    mma_bf16_16816(acc[mt][nt], c0.x, c1.x, c0.y, c1.y, bl[nt][0][0], bl[nt][0][1]);
                    mma_bf16_16816(acc[mt][nt], c0.z, c1.z, c0.w, c1.w, bl[nt][1][0], bl[nt][1][1]);
                } else {
                    mma_bf16_16816(acc[mt][nt], c0.x, c1.x, c0.y, c1.y, bh[nt][0][0], bh[nt][0][1]);
                    mma_bf16_16816(acc[mt][nt], c0.z, c1.z, c0.w, c1.w, bh[nt][1][0], bh[nt][1][1]);
                }
            }
        }
    }
    const float s = t.scale[t.a_slot[ja]];
    const int32_t o0 = t.soff[g.i], d = t.soff[g.i + 1] - o0;
    const int32_t col0 = kCB * g.ci + 8 * gq;
    if (col0 >= d) return;
    uint16_t *Y = a.y + o0 + col0;
    const uint32_t ysrc = wslot + kEBTile + 16 * lane;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        if (nt >= NT8) continue;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int32_t jt = kTGe * g.tg + 8 * nt + 2 * q + e;
            const int32_t tok = jt < L ? t.tok[p0 + jt] : -1;
            if (tok < 0) continue;
            const uint4 yv = lds16(ysrc + (2 * nt + e) * kChunk);
            uint4 o;
            o.x = pack_bf16x2(fmaf(s, acc[0][nt][e], bf16lo_to_f32(yv.x)), fmaf(s, acc[0][nt][2 + e], bf16hi_to_f32(yv.x)));
            o.y = pack_bf16x2(fmaf(s, acc[1][nt][e], bf16lo_to_f32(yv.y)), fmaf(s, acc[1][nt][2 + e], bf16hi_to_f32(yv.y)));
            o.z = pack_bf16x2(fmaf(s, acc[2][nt][e], bf16lo_to_f32(yv.z)), fmaf(s, acc[2][nt][2 + e], bf16hi_to_f32(yv.z)));
            o.w = pack_bf16x2(fmaf(s, acc[3][nt][e], bf16lo_to_f32(yv.w)), fmaf(s, acc[3][nt][2 + e], bf16hi_to_f32(yv.w)));
            stg_u4(Y + static_cast<int64_t>(tok) * a.ldy, o);
        }
    }
}

size_t direct_expand_smem(int32_t S, int32_t n, int32_t T) {
    return static_cast<size_t>(kEWarps) * kEStages * kESlot + tabs_bytes(S, n, T);
}

template <bool kF8>
__global__ void __launch_bounds__(32 * kEWarps, kECtas) direct_expand_kernel(DArgs a, Shape sh, const void *table) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[kEWarps][kEStages];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (lane == 0) {
        for (int s = 0; s < kEStages; ++s) mbar_init(sa(&bars[warp][s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const Tabs t = carve(smem + static_cast<size_t>(kEWarps) * kEStages * kESlot, sh.S, sh.n, a.T);
    // tables, B and y are not written by the shrink: read them before the wait
    if (a.plan != nullptr) load_plan<kF8>(a, sh, t, tabs_bytes(sh.S, sh.n, a.T));
    else build_tabs<true>(a, sh, table, t, VP<kF8>::BW, 1, 32);
    const float *buf = (t.misc[1] & 1) ? a.acc1 : a.acc0;
    const uint32_t wring = sa(smem) + warp * (kEStages * kESlot);
    EGen gi;
    e_first<kF8>(gi, t, sh.n);
    EGen gc = gi;
    // the whole ring in flight before the wait: B and y need nothing of the shrink
#pragma unroll
    for (int s = 0; s < kEStages; ++s) e_copy_stage<kF8>(gi, wring + s * kESlot, sa(&bars[warp][s]), t, sh, a, lane, sh.n);
    pdl_wait();
    float4 X[2][2][2];
    e_load_xa(gc, buf, t, sh, a.T, lane, X);
    int32_t it = 0;
    while (gc.live) {
        const int32_t sc = it % kEStages;
        EGen gn = gc;
        e_advance<kF8>(gn, t, sh.n);
        // the next unit's sums: the same registers while (slot, slice, token group) holds
        const bool same = gn.live && gn.ja == gc.ja && gn.i == gc.i && gn.tg == gc.tg;
        float4 Xn[2][2][2];
        if (!same) e_load_xa(gn, buf, t, sh, a.T, lane, Xn);
        cp_wait<kEStages - 1>();
        // a B tile that never lands (only a broken memory system) ends the warp's
        // walk: report it and issue nothing more into the ring
        if (!__all_sync(0xffffffffu, mbar_wait(sa(&bars[warp][sc]), static_cast<uint32_t>(it / kEStages) & 1u))) {
            if (lane == 0) report_error(a.err, LORA_ERR_TIMEOUT);
            break;
        }
        e_compute<kF8>(gc, wring + sc * kESlot, X, t, a, lane);
        __syncwarp();  // every lane's reads of slot sc are done: refill it with unit it + kEStages
        e_copy_stage<kF8>(gi, wring + sc * kESlot, sa(&bars[warp][sc]), t, sh, a, lane, sh.n);
        if (!same) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    X[nt][kb][0] = Xn[nt][kb][0];
                    X[nt][kb][1] = Xn[nt][kb][1];
                }
        }
        gc = gn;
        ++it;
    }
    cp_wait<0>();
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(a.exits, 1) == static_cast<int32_t>(gridDim.x) - 1) {
            *a.exits = 0;
            atomicAdd(a.gen, 1);
        }
    }
}

// A plan: the tables both kernels of a call would build in their prologue,
// built once for a batch (index) and shape by the same build_tabs and stored as
// two images, the shrink's then the expand's.  misc[2] records T, misc[6] the
// variant, misc[18] k and misc[19] r_max, which load_plan checks with the rest
// of the shape.  One launch builds the plans of up to
// kMaxPlanJobs slot tables of the same shape and batch (the layers of a step):
// block 2j + 0 / 2j + 1 writes the shrink / expand image of job j.
constexpr int kMaxPlanJobs = 120;
struct PlanJobs {
    const void *table[kMaxPlanJobs];
    unsigned char *plan[kMaxPlanJobs];
};

template <bool kF8>
__global__ void __launch_bounds__(256) direct_plan_kernel(DArgs a, Shape sh, PlanJobs jobs) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int job = blockIdx.x >> 1, img = blockIdx.x & 1;
    const void *table = jobs.table[job];
    unsigned char *plan = jobs.plan[job];
    const Tabs t = carve(smem, sh.S, sh.n, a.T);
    if (img == 0) build_tabs<false>(a, sh, table, t, VP<kF8>::TG, VP<kF8>::XF, VP<kF8>::BC);
    else build_tabs<true>(a, sh, table, t, VP<kF8>::BW, 1, 32);
    if (threadIdx.x == 0) {
        t.misc[2] = a.T;
        t.misc[6] = kF8 ? 1 : 0;
        t.misc[18] = sh.k;
        t.misc[19] = sh.r_max;
    }
    __syncthreads();
    const size_t bytes = tabs_bytes(sh.S, sh.n, a.T);
    unsigned char *out = plan + img * bytes;
    for (size_t o = 16 * static_cast<size_t>(threadIdx.x); o < bytes; o += 16 * static_cast<size_t>(blockDim.x))
        *reinterpret_cast<uint4 *>(out + o) = *reinterpret_cast<const uint4 *>(smem + o);
}

// Load-time scale of an FP8 B (TensorRT-LLM LoRA serving page, "第五步:FP8 特判"):
// w[e] = e4m3(clamp(bf16(value(w[e]) * scale), +-448)), the product exact in
// fp64 and rounded once to bf16; NaN codes become 0x7F.
__global__ void premultiply_e4m3_kernel(uint8_t *w, int64_t n, double scale) {
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint32_t h = f16x2_from_e4m3x2(w[e]);
        const double v = static_cast<double>(__half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xffffu))));
        const float b = __bfloat162float(__double2bfloat16(v * scale));
        uint32_t c;
        asm("{\n\t.reg .b16 p;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 p, %1, %1;\n\t"
            "cvt.u32.u16 %0, p;\n\t}"
            : "=r"(c) : "f"(b));
        w[e] = isnan(b) ? uint8_t(0x7F) : static_cast<uint8_t>(c & 0xffu);
    }
}

}  // namespace

cudaError_t launch_premultiply_e4m3(uint8_t *w, int64_t n, double scale, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
    premultiply_e4m3_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w, n, scale);
    return cudaGetLastError();
}

// fp8: A and B in float8_e4m3fn, whose rows of k bytes must stay 16-byte aligned.
bool decode_direct_supported(int32_t T, const Shape &sh, bool fp8) {
    return T >= 1 && T <= kMaxTokens && sh.r_max <= kMaxRank && sh.S <= kMaxSlots && sh.S * sh.n <= kMaxPtrs &&
           (!fp8 || sh.k % 16 == 0) && direct_shrink_smem(sh.S, sh.n, T) <= 227 * 1024 &&
           direct_expand_smem(sh.S, sh.n, T) <= 227 * 1024;  // past half an SM the grid runs in more waves
}

namespace {

cudaError_t direct_args(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                        const int32_t *sorted_ids, const int32_t *seg, const int32_t *active, float *ws, int32_t T,
                        int32_t *err, bool fp8, int32_t x_div, DArgs &a, int &num_sms) {
    if (!decode_direct_supported(T, sh, fp8)) return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const WorkspaceLayout W(T, sh.n, sh.r_max, sh.S);
    char *base = reinterpret_cast<char *>(ws);
    int32_t *ctrl = reinterpret_cast<int32_t *>(base);
    a.x = x;
    a.ldx = ldx;
    a.x_div = x_div;
    a.y = y;
    a.ldy = ldy;
    a.sorted_ids = sorted_ids;
    a.seg = seg;
    a.active = active;
    a.acc0 = reinterpret_cast<float *>(base + W.acc2_off);
    a.acc1 = reinterpret_cast<float *>(base + W.acc3_off);
    a.gen = ctrl + 2 * LORA_MAX_SLICES * static_cast<size_t>(sh.S);
    a.exits = a.gen + 1;
    a.err = err;
    a.T = T;
    a.plan = nullptr;
    return cudaSuccess;
}

}  // namespace

// A plan holds two table images (shrink, expand) of tabs_bytes each.
size_t direct_plan_bytes(int32_t T, const Shape &sh) { return 2 * tabs_bytes(sh.S, sh.n, T); }

// Builds the plans of `count` slot tables (one batch and shape) for the bf16 or
// the FP8 kernels, kMaxPlanJobs per launch.
cudaError_t launch_direct_plans(const Shape &sh, const void *const *tables, unsigned char *const *plans,
                                int32_t count, const int32_t *sorted_ids, const int32_t *seg, const int32_t *active,
                                int32_t T, bool fp8, int32_t *err, cudaStream_t stream) {
    if (!decode_direct_supported(T, sh, fp8)) return cudaErrorNotSupported;
    DArgs a = {};
    a.sorted_ids = sorted_ids;
    a.seg = seg;
    a.active = active;
    a.err = err;
    a.T = T;
    const size_t smem = tabs_bytes(sh.S, sh.n, T);
    auto kern = fp8 ? direct_plan_kernel<true> : direct_plan_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    for (int32_t j0 = 0; j0 < count; j0 += kMaxPlanJobs) {
        PlanJobs jobs = {};
        const int32_t m = std::min(kMaxPlanJobs, count - j0);
        for (int32_t j = 0; j < m; ++j) {
            jobs.table[j] = tables[j0 + j];
            jobs.plan[j] = plans[j0 + j];
        }
        kern<<<2 * m, 256, smem, stream>>>(a, sh, jobs);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// The x-only half: sums of x A^T into the call's buffer (reads x, A; writes the
// workspace only).  fp8: A is e4m3 and x is rounded to e4m3 on the way in.
cudaError_t launch_direct_shrink(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                 const void *table, const int32_t *sorted_ids, const int32_t *seg,
                                 const int32_t *active, float *ws, int32_t T, int32_t *err, bool fp8,
                                 cudaStream_t stream, int32_t x_div, const unsigned char *plan) {
    DArgs a;
    int num_sms = 0;
    cudaError_t e = direct_args(x, ldx, y, ldy, sh, sorted_ids, seg, active, ws, T, err, fp8, x_div, a, num_sms);
    if (e != cudaSuccess) return e;
    a.plan = plan;  // the shrink's image comes first
    const size_t s_smem = direct_shrink_smem(sh.S, sh.n, T);
    auto kern = fp8 ? direct_shrink_kernel<true> : direct_shrink_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s_smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(kSCtas * num_sms));
    cfg.blockDim = dim3(32 * kSWarps);
    cfg.dynamicSmemBytes = s_smem;
    cfg.stream = stream;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kern, a, sh, table);
}

// The y half: y += s (x A^T) B^T from the buffer the shrink of this call filled
// (fp8: B is e4m3).  `programmatic`: launched as a programmatic dependent of
// that shrink (it must then directly follow it on the stream).
cudaError_t launch_direct_expand(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                 const void *table, const int32_t *sorted_ids, const int32_t *seg,
                                 const int32_t *active, float *ws, int32_t T, int32_t *err, bool fp8,
                                 bool programmatic, cudaStream_t stream, const unsigned char *plan) {
    DArgs a;
    int num_sms = 0;
    cudaError_t e = direct_args(x, ldx, y, ldy, sh, sorted_ids, seg, active, ws, T, err, fp8, 1, a, num_sms);
    if (e != cudaSuccess) return e;
    a.plan = plan != nullptr ? plan + tabs_bytes(sh.S, sh.n, T) : nullptr;
    const size_t e_smem = direct_expand_smem(sh.S, sh.n, T);
    auto kern = fp8 ? direct_expand_kernel<true> : direct_expand_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(e_smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(kECtas * num_sms));
    cfg.blockDim = dim3(32 * kEWarps);
    cfg.dynamicSmemBytes = e_smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a, sh, table);
}

cudaError_t launch_decode_direct(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                 const void *table, const int32_t *sorted_ids, const int32_t *seg,
                                 const int32_t *active, float *ws, int32_t T, int32_t *err, bool fp8,
                                 cudaStream_t stream, int32_t x_div, const unsigned char *plan) {
    cudaError_t e = launch_direct_shrink(x, ldx, y, ldy, sh, table, sorted_ids, seg, active, ws, T, err, fp8,
                                         stream, x_div, plan);
    if (e != cudaSuccess) return e;
    return launch_direct_expand(x, ldx, y, ldy, sh, table, sorted_ids, seg, active, ws, T, err, fp8, true, stream,
                                plan);
}

}  // namespace lora
