// Fused single-launch decode path of the LoRA branch: shrink and expand in one
// persistent kernel.
//
// At decode the branch streams adapter weights: each active slot's A and B are
// read once while x and y are small (llama.cpp LoRA adapter page, section
// "为什么低秩增量可以「后加」": decode is bound by memory bandwidth and the
// branch's cost is extra launches and intermediates).  The kernel is built to
// keep HBM busy from a single launch:
//
//   * one CTA per SM (cooperative launch: all CTAs co-resident); a producer
//     warp streams the tiles of the CTA's work units into a 3-stage
//     shared-memory ring with TMA bulk copies (cp.async.bulk, completion counted
//     in bytes on an mbarrier); token rows of x, y and the accumulator are
//     gathered through sorted_ids, which the prologue keeps in shared memory;
//   * units are sized to about 48 KB of data, so a CTA runs a handful of them
//     and each SM keeps two to three units' bytes in flight;
//   * eight consumer warps run warp-level tensor-core MMA (bf16 in, fp32
//     accumulate) on the staged tiles, with up to three independent
//     accumulator chains per warp;
//   * shrink units are (slot, slice, <=64 rank rows, <=48 tokens, a k-chunk):
//     splitting k spreads the big slots' weights over all SMs (TensorRT-LLM LoRA
//     serving page, "path 2: split-K tuning"); partial sums are added into an
//     fp32 accumulator in the workspace with vector reductions
//     (red.global.add.v4.f32); each warp then arrives on a per-(slot, slice)
//     counter with release semantics;
//   * expand units are (slot, slice, a column chunk, <=48 tokens); the producer
//     copies their B and y tiles, waits (bounded) on the (slot, slice) counter,
//     then copies the finished accumulator rows, so consumers never wait across
//     CTAs;
//   * the last expand warp of a (slot, slice) zeroes its accumulator rows and
//     resets the counters, leaving the workspace ready for the next call.
//
// Every CTA issues and consumes all its shrink units before any expand unit,
// and shrink units wait on nothing outside their CTA, so every counter wait
// ends; all waits are still bounded (LORA_ERR_TIMEOUT) so that a bug cannot
// hang the GPU.  Limits of this path (the host routes other cases to the split
// kernels): T <= kMaxTokens, every rank <= kMaxRank.
#include <algorithm>

#include "common.cuh"

namespace lora {

namespace {

constexpr int kCWarps = 8;                          // consumer (MMA) warps
constexpr int kThreads = (kCWarps + 1) * 32;        // + one producer warp
constexpr int kStages = 3;
constexpr int kStageBytes = 64512;                  // one ring stage
constexpr int kTG = 48;                             // tokens per unit
constexpr int kRG = 64;                             // shrink: rank rows per unit
constexpr int kUnitBytes = 49152;                   // target data per unit
constexpr int kMaxTokens = 2048;                    // token ids kept in shared memory
constexpr int kMaxRank = 128;
constexpr int kILP = 3;                             // independent work items per warp
constexpr uint64_t kWaitNs = 50ull * 1000 * 1000;   // bound on any wait: 50 ms

__host__ __device__ inline int ceil_div_i(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int align128(int b) { return (b + 127) & ~127; }

// Shrink k-chunk for `rows` staged rows (rank rows + token rows): about
// kUnitBytes of data, a multiple of 64 columns, 64 at least.  Rows are stored
// with pitch kc*2 + 16 bytes (= 16 mod 128), so the eight 16-byte rows that one
// ldmatrix phase reads fall in eight different bank groups.
__device__ inline int shrink_kc(int rows, int k) {
    int kc = ((kUnitBytes / rows - 16) / 2) & ~63;
    const int kr = (k + 63) & ~63;
    kc = kc > kr ? kr : kc;
    return kc < 64 ? 64 : kc;
}

// Expand column chunk for rank r and up to `nt` tokens: B (cols x r bf16), y
// (nt rows of cols bf16, padded) and the accumulator rows (nt x r fp32, padded)
// within about kUnitBytes; a multiple of 32 columns, 32 at least.
__device__ inline int expand_cols(int r, int nt, int d_max) {
    const int acc = nt * (r * 4 + 16);
    int ec = ((kUnitBytes - acc - 64 * nt - 256) / (2 * r + 2 * nt)) & ~31;
    const int dr = (d_max + 31) & ~31;
    ec = ec > dr ? dr : ec;
    return ec < 32 ? 32 : ec;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase; false on timeout or when another warp of
// the CTA has aborted.  try_wait suspends the thread for a while in hardware;
// the timer and the abort flag are looked at every 256 polls only.
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

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// Shared-memory loads as plain C++ loads: the compiler schedules them freely
// and still keeps them after the mbarrier waits (asm volatile, "memory").
__device__ __forceinline__ uint4 lds128(const void *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ float4 lds_f4(const void *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ uint2 lds64(const void *p) { return *reinterpret_cast<const uint2 *>(p); }

// Four 8x8 bf16 matrices from shared memory; lane l supplies the row address
// of matrix l/8.  Volatile: it must stay after the mbarrier wait that made the
// stage's bytes visible.
__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(p)));
}

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ void red_add_release(int32_t *p, int32_t v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int32_t atom_add_acq_rel(int32_t *p, int32_t v) {
    int32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void stg_u2(void *p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(a), "r"(b) : "memory");
}

// ---------------------------------------------------------------------------
// Work units (everything read from the prologue's shared-memory tables)
// ---------------------------------------------------------------------------
struct Ctx {
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    const int32_t *sorted_ids;
    const int32_t *seg;
    int32_t *shrink_done;   // [S][LORA_MAX_SLICES]
    int32_t *expand_done;   // [S][LORA_MAX_SLICES]
    float *acc;             // [n][T][r_max]
    int32_t *err;
    int32_t T;
};

struct Tables {
    const int32_t *seg;     // [S + 2]
    const int32_t *rank;    // [S]
    const int32_t *pref_s;  // [S] exclusive prefix of shrink units
    const int32_t *pref_e;  // [S] exclusive prefix of expand units
    const int32_t *tok;     // [T] sorted_ids
};


__device__ __forceinline__ int slice_width_max(const Shape &sh) {
    int d = 0;
    for (int i = 0; i < sh.n; ++i) d = max(d, sh.off[i + 1] - sh.off[i]);
    return d;
}

struct ShrinkUnit {
    int s, i, rg, p0, n, r, R, tok0, ntok, kc0, W, pitch;
};

struct ExpandUnit {
    int s, i, p0, n, r, tok0, ntok, c0, EW, EC, TGs, y_off, acc_off, ypitch, apitch;
};

// A unit reduced to its indices; the geometry follows with multiplies only.
// a = rank group (shrink) or column chunk (expand); b = k-chunk (shrink);
// size = k-chunk width (shrink) or column chunk width (expand).
struct UnitIdx {
    int32_t s;
    int16_t kind, i, a, tg;
    int32_t b, size;
};

constexpr int kMaxUnits = 128;  // unit indices kept in shared memory per CTA

// Rows a shrink unit of this slot may read: its rank rows, then its token rows
// rounded up to the 16-row ldmatrix tiles (the A tile's own rounding to 16
// rows stays inside this bound).  The k-chunk is sized from it, so every
// fragment read stays inside the stage.
__device__ __forceinline__ int shrink_rows(int n, int r) { return min(r, kRG) + 16 * ceil_div_i(min(n, kTG), 16); }

__device__ __forceinline__ int shrink_units_of(int n, int r, const Shape &sh) {
    const int kc = shrink_kc(shrink_rows(n, r), sh.k);
    return sh.n * ceil_div_i(r, kRG) * ceil_div_i(n, kTG) * ceil_div_i(sh.k, kc);
}

__device__ __forceinline__ int expand_units_of(int n, int r, const Shape &sh) {
    const int ec = expand_cols(r, min(n, kTG), slice_width_max(sh));
    int c = 0;
    for (int i = 0; i < sh.n; ++i) c += ceil_div_i(sh.off[i + 1] - sh.off[i], ec);
    return c * ceil_div_i(n, kTG);
}

// The full decode (integer divisions); run once per unit, in parallel, in the prologue.
__device__ UnitIdx decode_unit(int32_t v, int32_t NS, const Tables &tb, const Shape &sh) {
    UnitIdx x;
    if (v < NS) {
        x.kind = 0;
        x.s = find_slot(tb.pref_s, sh.S, v);
        int32_t l = v - tb.pref_s[x.s];
        const int n = tb.seg[x.s + 1] - tb.seg[x.s], r = tb.rank[x.s];
        const int kc = shrink_kc(shrink_rows(n, r), sh.k);
        const int RGs = ceil_div_i(r, kRG), TGs = ceil_div_i(n, kTG), KCs = ceil_div_i(sh.k, kc);
        x.b = l % KCs;
        l /= KCs;
        x.tg = static_cast<int16_t>(l % TGs);
        l /= TGs;
        x.a = static_cast<int16_t>(l % RGs);
        x.i = static_cast<int16_t>(l / RGs);
        x.size = kc;
    } else {
        v -= NS;
        x.kind = 1;
        x.s = find_slot(tb.pref_e, sh.S, v);
        int32_t l = v - tb.pref_e[x.s];
        const int n = tb.seg[x.s + 1] - tb.seg[x.s], r = tb.rank[x.s];
        const int ec = expand_cols(r, min(n, kTG), slice_width_max(sh));
        const int TGs = ceil_div_i(n, kTG);
        x.tg = static_cast<int16_t>(l % TGs);
        l /= TGs;
        int i = 0;
        while (i < sh.n - 1) {
            const int nc = ceil_div_i(sh.off[i + 1] - sh.off[i], ec);
            if (l < nc) break;
            l -= nc;
            ++i;
        }
        x.i = static_cast<int16_t>(i);
        x.a = static_cast<int16_t>(l);
        x.b = 0;
        x.size = ec;
    }
    return x;
}

__device__ __forceinline__ ShrinkUnit make_shrink(const UnitIdx &x, const Tables &tb, const Shape &sh) {
    ShrinkUnit w;
    w.s = x.s;
    w.i = x.i;
    w.rg = x.a;
    w.p0 = tb.seg[x.s];
    w.n = tb.seg[x.s + 1] - w.p0;
    w.r = tb.rank[x.s];
    w.R = min(kRG, w.r - w.rg * kRG);
    w.tok0 = x.tg * kTG;
    w.ntok = min(kTG, w.n - w.tok0);
    w.kc0 = x.b * x.size;
    w.W = min(x.size, sh.k - w.kc0);
    w.pitch = x.size * 2 + 16;
    return w;
}

__device__ __forceinline__ ExpandUnit make_expand(const UnitIdx &x, const Tables &tb, const Shape &sh) {
    ExpandUnit e;
    e.s = x.s;
    e.i = x.i;
    e.p0 = tb.seg[x.s];
    e.n = tb.seg[x.s + 1] - e.p0;
    e.r = tb.rank[x.s];
    e.EC = x.size;
    e.TGs = ceil_div_i(e.n, kTG);
    e.c0 = x.a * e.EC;
    e.EW = min(e.EC, sh.off[e.i + 1] - sh.off[e.i] - e.c0);
    e.tok0 = x.tg * kTG;
    e.ntok = min(kTG, e.n - e.tok0);
    e.ypitch = e.EC * 2 + 64;
    e.apitch = e.r * 4 + 16;
    e.y_off = align128(e.EC * e.r * 2);
    e.acc_off = align128(e.y_off + min(e.n, kTG) * e.ypitch);
    return e;
}

// a / b for 0 <= a < 2^20 and 1 <= b <= 2^10, exactly: (a + 1/2) / b is at
// least 1/(2b) away from an integer, far above the float rounding error.
__device__ __forceinline__ int div_small(int a, int b) {
    return __float2int_rz((static_cast<float>(a) + 0.5f) * __frcp_rn(static_cast<float>(b)));
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) fused_decode_kernel(Ctx c, Shape sh, const void *__restrict__ table) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;                                                  // kStages x kStageBytes
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + kStages * kStageBytes);  // [kStages]
    uint64_t *empty = full + kStages;                                            // [kStages]
    float *scratch = reinterpret_cast<float *>(empty + kStages);                 // [kCWarps][16 x 16]
    int32_t *s_seg = reinterpret_cast<int32_t *>(scratch + kCWarps * 256);      // [S + 2]
    int32_t *s_rank = s_seg + sh.S + 2;                                          // [S]
    int32_t *pref_s = s_rank + sh.S;                                             // [S]
    int32_t *pref_e = pref_s + sh.S;                                             // [S]
    int32_t *s_tok = pref_e + sh.S;                                              // [T]
    int32_t *scan_scr = s_tok + c.T;                                             // [33]
    volatile int32_t *abort_flag = scan_scr + 33;                                // [1]
    UnitIdx *s_units = reinterpret_cast<UnitIdx *>(scan_scr + 40);              // [kMaxUnits]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
    const TableView tab(table, sh.S, sh.n);

    // ---------------------------------------------------------------- prologue
    const int32_t *hdr = static_cast<const int32_t *>(table);
    const bool ok = hdr[0] == kTableMagic && hdr[1] == sh.S && hdr[2] == sh.n && c.seg[sh.S + 1] == c.T;
    if (!ok && tid == 0 && blockIdx.x == 0) report_error(c.err, LORA_ERR_INVALID_ARG);
    for (int e = tid; e < sh.S + 2; e += blockDim.x) s_seg[e] = ok ? c.seg[e] : 0;
    for (int e = tid; e < c.T; e += blockDim.x) s_tok[e] = c.sorted_ids[e];
    for (int s = tid; s < sh.S; s += blockDim.x) {
        const int r = ok ? tab.rank[s] : 0;
        const bool rank_ok = r <= sh.r_max && r <= kMaxRank;
        if (!rank_ok && blockIdx.x == 0) report_error(c.err, LORA_ERR_RANK);
        s_rank[s] = rank_ok ? r : 0;
    }
    if (tid == 0) {
        *abort_flag = 0;
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kCWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    for (int s = tid; s < sh.S; s += blockDim.x) {
        const int n = s_seg[s + 1] - s_seg[s];
        const int r = s_rank[s];
        const bool act = n > 0 && r > 0;
        pref_s[s] = act ? shrink_units_of(n, r, sh) : 0;
        pref_e[s] = act ? expand_units_of(n, r, sh) : 0;
    }
    __syncthreads();
    const int32_t NS = block_exclusive_scan(pref_s, sh.S, scan_scr);
    const int32_t NE = block_exclusive_scan(pref_e, sh.S, scan_scr);
    const Tables tb{s_seg, s_rank, pref_s, pref_e, s_tok};
    const int32_t G = gridDim.x, b = blockIdx.x;
    // this CTA's units: shrink b, b+G, ..., then expand b, b+G, ...
    const int32_t my_s = NS > b ? ceil_div_i(NS - b, G) : 0;
    const int32_t my_e = NE > b ? ceil_div_i(NE - b, G) : 0;
    const int32_t my_total = my_s + my_e;
    // decode this CTA's units once, in parallel (unit j of this CTA is global unit
    // b + j*G among shrink units, then b + (j - my_s)*G among expand units)
    for (int j = tid; j < min(my_total, kMaxUnits); j += blockDim.x) {
        const int32_t v = j < my_s ? b + j * G : NS + b + (j - my_s) * G;
        s_units[j] = decode_unit(v, NS, tb, sh);
    }
    __syncthreads();
    auto unit_at = [&](int32_t j) -> UnitIdx {
        if (j < kMaxUnits) return s_units[j];
        return decode_unit(j < my_s ? b + j * G : NS + b + (j - my_s) * G, NS, tb, sh);
    };

    if (warp == kCWarps) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t parity = 1;  // the first pass over the ring does not wait
        int32_t issued = 0;
        for (int32_t it = 0; it < my_total; ++it) {
            bool got = true;
            if (lane == 0) got = mbar_wait(&empty[stage], parity, abort_flag);
            got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!got) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report_error(c.err, LORA_ERR_TIMEOUT);
                }
                break;
            }
            unsigned char *st = ring + stage * kStageBytes;
            if (it < my_s) {
                const ShrinkUnit w = make_shrink(unit_at(it), tb, sh);
                const uint32_t row_bytes = static_cast<uint32_t>(w.W) * 2u;
                if (lane == 0) mbar_arrive_expect_tx(&full[stage], row_bytes * static_cast<uint32_t>(w.R + w.ntok));
                __syncwarp();
                const uint16_t *A = reinterpret_cast<const uint16_t *>(tab.a_ptr[w.s * sh.n + w.i]);
                for (int j = lane; j < w.R + w.ntok; j += 32) {
                    const uint16_t *src;
                    if (j < w.R) src = A + static_cast<int64_t>(w.rg * kRG + j) * sh.k + w.kc0;
                    else src = c.x + static_cast<int64_t>(s_tok[w.p0 + w.tok0 + j - w.R]) * c.ldx + w.kc0;
                    bulk_g2s(st + j * w.pitch, src, row_bytes, &full[stage]);
                }
            } else {
                const ExpandUnit e = make_expand(unit_at(it), tb, sh);
                const uint32_t b_bytes = static_cast<uint32_t>(e.EW) * static_cast<uint32_t>(e.r) * 2u;
                const uint32_t y_bytes = static_cast<uint32_t>(e.EW) * 2u;
                const uint32_t a_bytes = static_cast<uint32_t>(e.r) * 4u;
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[stage], b_bytes + (y_bytes + a_bytes) * static_cast<uint32_t>(e.ntok));
                __syncwarp();
                if (lane == 0) {
                    const uint16_t *B = reinterpret_cast<const uint16_t *>(tab.b_ptr[e.s * sh.n + e.i]);
                    bulk_g2s(st, B + static_cast<int64_t>(e.c0) * e.r, b_bytes, &full[stage]);
                }
                for (int tt = lane; tt < e.ntok; tt += 32) {
                    const int32_t t = s_tok[e.p0 + e.tok0 + tt];
                    bulk_g2s(st + e.y_off + tt * e.ypitch, c.y + static_cast<int64_t>(t) * c.ldy + sh.off[e.i] + e.c0,
                             y_bytes, &full[stage]);
                }
                // the accumulator rows are final once every shrink warp of this
                // (slot, slice) has arrived on its counter
                if (lane == 0) {
                    const int32_t need = kCWarps * e.TGs * ceil_div_i(e.r, kRG) *
                                         ceil_div_i(sh.k, shrink_kc(shrink_rows(e.n, e.r), sh.k));
                    const uint64_t t0 = globaltimer_ns();
                    int spin = 0;
                    while (ld_acquire(&c.shrink_done[e.s * LORA_MAX_SLICES + e.i]) < need) {
                        if ((++spin & 63) == 0 && globaltimer_ns() - t0 > kWaitNs) {
                            report_error(c.err, LORA_ERR_TIMEOUT);  // copy anyway: the barrier still completes
                            break;
                        }
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");  // generic writes -> async reads
                }
                __syncwarp();
                const float *acc_rows = c.acc + static_cast<int64_t>(e.i) * c.T * sh.r_max;
                for (int tt = lane; tt < e.ntok; tt += 32) {
                    const int32_t t = s_tok[e.p0 + e.tok0 + tt];
                    bulk_g2s(st + e.acc_off + tt * e.apitch, acc_rows + static_cast<int64_t>(t) * sh.r_max, a_bytes,
                             &full[stage]);
                }
            }
            ++issued;
            if (++stage == kStages) {
                stage = 0;
                parity ^= 1u;
            }
        }
        // On abort, copies already issued must land before the CTA exits: wait
        // (bounded) for the last phase of every stage that was filled.
        if (lane == 0 && *abort_flag) {
            for (int32_t it = max(0, issued - kStages); it < issued; ++it) {
                const uint64_t t0 = globaltimer_ns();
                const uint32_t ph = static_cast<uint32_t>((it / kStages) & 1);
                while (!mbar_try_wait(&full[it % kStages], ph) && globaltimer_ns() - t0 < kWaitNs) {
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    float *scr = scratch + warp * 256;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    int stage = 0;
    uint32_t parity = 0;
    for (int32_t it = 0; it < my_total; ++it) {
        if (!mbar_wait(&full[stage], parity, abort_flag)) {
            if (lane == 0) {
                *abort_flag = 1;
                report_error(c.err, LORA_ERR_TIMEOUT);
            }
            break;
        }
        const unsigned char *st = ring + stage * kStageBytes;
        if (it < my_s) {
            // ------------------------------------------------------- shrink unit
            // items: (16 rank rows) x (16 tokens) output tiles, times a split of the
            // k-steps over warps when there are few tiles; up to kILP items per warp
            // run together.  Fragments come from ldmatrix (standard m16n8k16 layout).
            const ShrinkUnit w = make_shrink(unit_at(it), tb, sh);
            const int nb = ceil_div_i(w.R, 16), ntp = ceil_div_i(w.ntok, 16), ksteps = w.W >> 4;
            const int tiles = nb * ntp;
            const int ksplit = max(1, min(kCWarps / tiles, ksteps));
            const int items = tiles * ksplit;
            const unsigned char *sA = st, *sX = st + w.R * w.pitch;
            // per-lane ldmatrix row offsets (bytes) inside a 16-row block at k-step 0
            const int a_lane = (lane & 15) * w.pitch + (lane >> 4) * 16;
            const int x_lane = ((lane & 7) + ((lane >> 4) << 3)) * w.pitch + ((lane >> 3) & 1) * 16;
            for (int base = warp; base < items; base += kCWarps * kILP) {
                float acc[kILP][2][4];
                int rbm[kILP], tpm[kILP], k0[kILP], len[kILP];
                int maxlen = 0;
#pragma unroll
                for (int m = 0; m < kILP; ++m) {
                    const int item = base + m * kCWarps;
#pragma unroll
                    for (int u = 0; u < 2; ++u) acc[m][u][0] = acc[m][u][1] = acc[m][u][2] = acc[m][u][3] = 0.f;
                    const int tile = div_small(item, ksplit), ks = item - tile * ksplit;
                    tpm[m] = div_small(tile, nb);
                    rbm[m] = tile - tpm[m] * nb;
                    k0[m] = div_small(ks * ksteps, ksplit);
                    len[m] = item < items ? div_small((ks + 1) * ksteps, ksplit) - k0[m] : 0;
                    maxlen = max(maxlen, len[m]);
                }
                for (int step = 0; step < maxlen; ++step) {
                    uint32_t a[kILP][4], xb[kILP][4];
#pragma unroll
                    for (int m = 0; m < kILP; ++m) {
                        if (step < len[m]) {
                            const int kb = (k0[m] + step) * 32;  // byte offset of this k-step in a row
                            ldsm_x4(sA + rbm[m] * 16 * w.pitch + a_lane + kb, a[m][0], a[m][1], a[m][2], a[m][3]);
                            ldsm_x4(sX + tpm[m] * 16 * w.pitch + x_lane + kb, xb[m][0], xb[m][1], xb[m][2], xb[m][3]);
                        }
                    }
#pragma unroll
                    for (int m = 0; m < kILP; ++m) {
                        if (step < len[m]) {
                            mma_bf16_16816(acc[m][0], a[m][0], a[m][1], a[m][2], a[m][3], xb[m][0], xb[m][1]);
                            mma_bf16_16816(acc[m][1], a[m][0], a[m][1], a[m][2], a[m][3], xb[m][2], xb[m][3]);
                        }
                    }
                }
                // transpose each 16 x 16 partial to [token][rank] and add 4 ranks at a time
#pragma unroll
                for (int m = 0; m < kILP; ++m) {
                    if (len[m] == 0) continue;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        scr[(8 * u + 2 * q) * 16 + g] = acc[m][u][0];
                        scr[(8 * u + 2 * q + 1) * 16 + g] = acc[m][u][1];
                        scr[(8 * u + 2 * q) * 16 + g + 8] = acc[m][u][2];
                        scr[(8 * u + 2 * q + 1) * 16 + g + 8] = acc[m][u][3];
                    }
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int idx = lane + 32 * h;             // 16 tokens x 4 rank quads
                        const int tl = idx >> 2, jq = idx & 3;
                        const int tk = tpm[m] * 16 + tl, row = rbm[m] * 16 + 4 * jq;
                        if (tk < w.ntok && row < w.R) {
                            const float4 v = *reinterpret_cast<const float4 *>(scr + tl * 16 + 4 * jq);
                            const int32_t t = s_tok[w.p0 + w.tok0 + tk];
                            red_add_v4(c.acc + (static_cast<int64_t>(w.i) * c.T + t) * sh.r_max + w.rg * kRG + row,
                                       v.x, v.y, v.z, v.w);
                        }
                    }
                    __syncwarp();
                }
            }
            // this warp's reductions precede its arrival on the counter:
            // __syncwarp orders the lanes, the release increment publishes them
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[stage]);
                red_add_release(&c.shrink_done[w.s * LORA_MAX_SLICES + w.i], 1);
            }
        } else {
            // ------------------------------------------------------- expand unit
            const ExpandUnit e = make_expand(unit_at(it), tb, sh);
            const int nt8 = e.EW / 8, npairs = ceil_div_i(nt8, 2), ntt = ceil_div_i(e.ntok, 16);
            const int items = ntt * npairs;
            const int ctr = e.s * LORA_MAX_SLICES + e.i;
            const unsigned char *sB = st, *sY = st + e.y_off, *sAcc = st + e.acc_off;
            const float scale = tab.scale[e.s];
            const int kbn = ceil_div_i(e.r, 32);
            for (int base = warp; base < items; base += kCWarps * kILP) {
                float acc[kILP][2][4];
                int ttm[kILP], pairm[kILP];
                bool val[kILP];
#pragma unroll
                for (int m = 0; m < kILP; ++m) {
                    const int item = base + m * kCWarps;
                    val[m] = item < items;
                    ttm[m] = div_small(item, npairs);
                    pairm[m] = item - ttm[m] * npairs;
#pragma unroll
                    for (int u = 0; u < 2; ++u) acc[m][u][0] = acc[m][u][1] = acc[m][u][2] = acc[m][u][3] = 0.f;
                }
                for (int kb = 0; kb < kbn; ++kb) {
                    const int j = kb * 32 + 8 * q;
                    const bool jok = j < e.r;
                    uint4 ha[kILP], la[kILP], hb[kILP], lb[kILP], bv[kILP][2];
#pragma unroll
                    for (int m = 0; m < kILP; ++m) {
                        const int ra = ttm[m] * 16 + g, rb2 = ra + 8;
                        // A operand: accumulator rows g (ra) and g+8 (rb2), ranks j..j+7, as bf16 hi + lo
                        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
                        if (val[m] && jok && ra < e.ntok) {
                            a0 = lds_f4(sAcc + ra * e.apitch + j * 4);
                            a1 = lds_f4(sAcc + ra * e.apitch + j * 4 + 16);
                        }
                        if (val[m] && jok && rb2 < e.ntok) {
                            b0 = lds_f4(sAcc + rb2 * e.apitch + j * 4);
                            b1 = lds_f4(sAcc + rb2 * e.apitch + j * 4 + 16);
                        }
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            // n-tile u of the pair: the lane's B row is column 16*pair + 4*(g/2) + 2u + g%2,
                            // so its outputs land on columns 16*pair + 4q + 2u + {0, 1}
                            const int col = pairm[m] * 16 + 4 * (g >> 1) + 2 * u + (g & 1);
                            bv[m][u] = (val[m] && jok && col < e.EW) ? lds128(sB + (col * e.r + j) * 2) : z;
                        }
                        split_bf16x2(a0.x, a0.y, ha[m].x, la[m].x);
                        split_bf16x2(a0.z, a0.w, ha[m].y, la[m].y);
                        split_bf16x2(a1.x, a1.y, ha[m].z, la[m].z);
                        split_bf16x2(a1.z, a1.w, ha[m].w, la[m].w);
                        split_bf16x2(b0.x, b0.y, hb[m].x, lb[m].x);
                        split_bf16x2(b0.z, b0.w, hb[m].y, lb[m].y);
                        split_bf16x2(b1.x, b1.y, hb[m].z, lb[m].z);
                        split_bf16x2(b1.z, b1.w, hb[m].w, lb[m].w);
                    }
#pragma unroll
                    for (int m = 0; m < kILP; ++m) {
                        if (!val[m]) continue;
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            mma_bf16_16816(acc[m][u], ha[m].x, hb[m].x, ha[m].y, hb[m].y, bv[m][u].x, bv[m][u].y);
                            mma_bf16_16816(acc[m][u], la[m].x, lb[m].x, la[m].y, lb[m].y, bv[m][u].x, bv[m][u].y);
                        }
                    }
#pragma unroll
                    for (int m = 0; m < kILP; ++m) {
                        if (!val[m]) continue;
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            mma_bf16_16816(acc[m][u], ha[m].z, hb[m].z, ha[m].w, hb[m].w, bv[m][u].z, bv[m][u].w);
                            mma_bf16_16816(acc[m][u], la[m].z, lb[m].z, la[m].w, lb[m].w, bv[m][u].z, bv[m][u].w);
                        }
                    }
                }
                // y = y + scale * acc with one rounding; the lane owns 4 consecutive columns
#pragma unroll
                for (int m = 0; m < kILP; ++m) {
                    if (!val[m]) continue;
                    const int col0 = pairm[m] * 16 + 4 * q;
                    if (col0 >= e.EW) continue;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int row = ttm[m] * 16 + g + 8 * half;
                        if (row >= e.ntok) continue;
                        const int32_t t = s_tok[e.p0 + e.tok0 + row];
                        const uint2 yv = lds64(sY + row * e.ypitch + col0 * 2);
                        const float v0 = fmaf(scale, acc[m][0][2 * half + 0], bf16lo_to_f32(yv.x));
                        const float v1 = fmaf(scale, acc[m][0][2 * half + 1], bf16hi_to_f32(yv.x));
                        const float v2 = fmaf(scale, acc[m][1][2 * half + 0], bf16lo_to_f32(yv.y));
                        const float v3 = fmaf(scale, acc[m][1][2 * half + 1], bf16hi_to_f32(yv.y));
                        stg_u2(c.y + static_cast<int64_t>(t) * c.ldy + sh.off[e.i] + e.c0 + col0, pack_bf16x2(v0, v1),
                               pack_bf16x2(v2, v3));
                    }
                }
            }
            __syncwarp();
            int32_t old = 0;
            if (lane == 0) {
                mbar_arrive(&empty[stage]);
                old = atom_add_acq_rel(&c.expand_done[ctr], 1);
            }
            old = __shfl_sync(0xffffffffu, old, 0);
            // expand warps of this (slot, slice): kCWarps per unit, units = column chunks x token groups
            const int32_t e_need = kCWarps * ceil_div_i(sh.off[e.i + 1] - sh.off[e.i], e.EC) * e.TGs;
            if (old == e_need - 1) {
                // the last reader of this (slot, slice): clear its accumulator rows and both counters
                const int r4 = e.r / 4;
                float *acc_rows = c.acc + static_cast<int64_t>(e.i) * c.T * sh.r_max;
                for (int idx = lane; idx < e.n * r4; idx += 32) {
                    const int tk = idx / r4, j4 = idx % r4;
                    *reinterpret_cast<float4 *>(acc_rows + static_cast<int64_t>(s_tok[e.p0 + tk]) * sh.r_max + 4 * j4) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (lane == 0) {
                    c.shrink_done[ctr] = 0;
                    c.expand_done[ctr] = 0;
                }
            }
        }
        if (++stage == kStages) {
            stage = 0;
            parity ^= 1u;
        }
    }
}

size_t fused_smem_bytes(int32_t S, int32_t T) {
    return size_t(kStages) * kStageBytes + 2 * kStages * sizeof(uint64_t) + kCWarps * 256 * sizeof(float) +
           sizeof(int32_t) * (4 * size_t(S) + 2 + size_t(T) + 40) + kMaxUnits * sizeof(UnitIdx);
}

}  // namespace

bool fused_decode_supported(int32_t T, int32_t r_max, int32_t k) {
    return T <= kMaxTokens && r_max <= kMaxRank && k % 16 == 0;
}

cudaError_t launch_fused_decode(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                const void *table, const int32_t *sorted_ids, const int32_t *seg, float *ws,
                                int32_t T, int32_t *err, cudaStream_t stream) {
    if (!fused_decode_supported(T, sh.r_max, sh.k)) return cudaErrorNotSupported;
    // per call: the SM count and the attribute belong to the current device
    int dev = 0, num_sms = 0;
    {
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const size_t max_smem = fused_smem_bytes(LORA_MAX_SLOTS, kMaxTokens);
        e = cudaFuncSetAttribute(fused_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(max_smem));
        if (e != cudaSuccess) return e;
    }
    const WorkspaceLayout L(T, sh.n, sh.r_max, sh.S);
    char *base = reinterpret_cast<char *>(ws);
    Ctx c;
    c.x = x;
    c.ldx = ldx;
    c.y = y;
    c.ldy = ldy;
    c.sorted_ids = sorted_ids;
    c.seg = seg;
    c.shrink_done = reinterpret_cast<int32_t *>(base);
    c.expand_done = c.shrink_done + size_t(sh.S) * LORA_MAX_SLICES;
    c.acc = reinterpret_cast<float *>(base + L.acc_off);
    c.err = err;
    c.T = T;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = fused_smem_bytes(sh.S, T);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_decode_kernel, c, sh, table);
}

}  // namespace lora
