// Fused single-launch decode path of the LoRA branch: shrink and expand in one
// persistent kernel.
//
// The branch at decode streams adapter weights: each active slot's A and B are
// read once while x and y are small (llama.cpp LoRA adapter page, section
// "为什么低秩增量可以「后加」": decode is bound by memory bandwidth, the branch's
// cost is extra launches and intermediates).  So the kernel is built around
// keeping HBM busy:
//
//   * one CTA per SM; a producer warp streams the tiles of this CTA's work
//     units into a 3-stage shared-memory ring with TMA bulk copies
//     (cp.async.bulk + mbarrier transaction counts), one copy per tile row;
//     token rows of x and y are gathered through sorted_ids;
//   * eight consumer warps run warp-level tensor-core MMA (bf16 in, fp32
//     accumulate) on the staged tiles;
//   * shrink units are (slot, slice, 64 rank rows, 48 tokens, 256 of k): the
//     split over k gives every SM a share of the big slots' weights
//     (TensorRT-LLM LoRA serving page, "path 2: split-K tuning"); partial
//     results are added into an fp32 accumulator in the workspace with vector
//     reductions (red.global.add.v4.f32);
//   * expand units are (slot, slice, up to 128 output columns, 48 tokens);
//     their B and y tiles are prefetched while shrink units still run; before
//     reading the accumulator a warp waits (bounded) until every shrink unit of
//     its (slot, slice) has arrived on a per-(slot, slice) counter;
//   * the last expand warp of a (slot, slice) zeroes its accumulator rows and
//     resets both counters, so the workspace is ready for the next call with
//     no separate clearing launch.
//
// All CTAs are co-resident (cooperative launch) and every CTA finishes its
// shrink units before it waits on any counter, so the waits always end; they
// are still bounded (LORA_ERR_TIMEOUT) so that a bug can never hang the GPU.
#include <algorithm>

#include "common.cuh"

namespace lora {

namespace {

constexpr int kCWarps = 8;                          // consumer (MMA) warps
constexpr int kThreads = (kCWarps + 1) * 32;        // + one producer warp
constexpr int kStages = 3;
constexpr int kKC = 256;                            // shrink: k columns per unit
constexpr int kTG = 48;                             // tokens per unit (6 n-tiles of 8)
constexpr int kRG = 64;                             // shrink: rank rows per unit
constexpr int kPitch = kKC * 2 + 64;                // smem row pitch of shrink tiles (bytes)
constexpr int kStageBytes = (kRG + kTG) * kPitch;   // 64512
constexpr int kBTileBytes = 16384;                  // expand: B tile (<= 128 cols x 64 ranks)
constexpr uint64_t kWaitNs = 50ull * 1000 * 1000;   // bound on any wait: 50 ms

static_assert(kStageBytes % 128 == 0, "stage alignment");

// Expand column chunk for rank r: 128 columns up to r = 64, fewer above, so the
// B tile stays within kBTileBytes; always a multiple of 32 (16-byte aligned
// TMA addresses for every chunk).
__host__ __device__ inline int expand_cols(int r) {
    int ec = (8192 / (r < 64 ? 64 : r)) & ~31;
    return ec < 32 ? 32 : (ec > 128 ? 128 : ec);
}

// Row pitch (bytes) of a bf16 tile of r columns read 16 bytes per lane by MMA
// fragments: pitch / 4 = 16 (mod 32) puts two consecutive rows in different
// bank halves, so a quarter-warp's reads are conflict-free.
__device__ __forceinline__ int frag_pitch(int r) {
    int p = r * 2;
    while (((p >> 2) & 31) != 16) p += 16;
    return p;
}

constexpr int kAccOff = 32768;     // expand: staged accumulator (hi, lo) tiles
constexpr int kAccStageMaxR = 128; // ranks up to this are staged through shared memory

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy wrappers
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

// Bounded wait on an mbarrier phase; false on timeout or when another warp
// has aborted the CTA.
__device__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int32_t *abort_flag,
                          uint64_t limit_ns = kWaitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ uint2 lds64(const void *p) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ int32_t atom_add_acq_rel(int32_t *p, int32_t v) {
    int32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void stg_u2(void *p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(a), "r"(b) : "memory");
}

// Barrier among the consumer warps, on an mbarrier so the wait is bounded: if a
// warp has aborted, the others give up instead of waiting forever.  Each warp
// keeps its own phase bit.  Returns false on timeout or abort.
__device__ __forceinline__ bool consumer_barrier(uint64_t *bar, uint32_t &phase, volatile int32_t *abort_flag) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    // longer than the cross-CTA counter wait of the warp that arrives last
    const bool ok = mbar_wait(bar, phase, abort_flag, 3 * kWaitNs);
    phase ^= 1u;
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0 && ok;
}

__device__ __forceinline__ void sts64(void *p, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.u32 [%0], {%1,%2};" :: "r"(smem_u32(p)), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void split_bf16x2(float v0, float v1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16x2(v0, v1);
    lo = pack_bf16x2(v0 - bf16lo_to_f32(hi), v1 - bf16hi_to_f32(hi));
}

// ---------------------------------------------------------------------------
// Work units
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

struct SlotGeom {
    int s, p0, n, r, TGs;
};

__device__ __forceinline__ int32_t find_slot(const int32_t *pref, int32_t S, int32_t u) {
    int32_t lo = 0, hi = S;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (pref[mid] <= u) lo = mid + 1;
        else hi = mid;
    }
    return lo - 1;
}

struct ShrinkUnit {
    int s, i, rg, p0, n, r, R, tok0, ntok, kc0, W;
};

struct ExpandUnit {
    int s, i, p0, n, r, tok0, ntok, c0, EW, EC;
};

__device__ ShrinkUnit decode_shrink(int32_t u, const int32_t *pref, const Shape &sh, const TableView &tab,
                                    const int32_t *seg) {
    ShrinkUnit w;
    w.s = find_slot(pref, sh.S, u);
    int32_t l = u - pref[w.s];
    w.p0 = seg[w.s];
    w.n = seg[w.s + 1] - w.p0;
    w.r = tab.rank[w.s];
    const int RG = ceil_div_i(w.r, kRG), TGs = ceil_div_i(w.n, kTG), KCs = ceil_div_i(sh.k, kKC);
    const int kc = l % KCs;
    l /= KCs;
    const int tg = l % TGs;
    l /= TGs;
    w.rg = l % RG;
    w.i = l / RG;
    w.R = min(kRG, w.r - w.rg * kRG);
    w.tok0 = tg * kTG;
    w.ntok = min(kTG, w.n - w.tok0);
    w.kc0 = kc * kKC;
    w.W = min(kKC, sh.k - w.kc0);
    return w;
}

__device__ ExpandUnit decode_expand(int32_t v, const int32_t *pref, const Shape &sh, const TableView &tab,
                                    const int32_t *seg) {
    ExpandUnit e;
    e.s = find_slot(pref, sh.S, v);
    int32_t l = v - pref[e.s];
    e.p0 = seg[e.s];
    e.n = seg[e.s + 1] - e.p0;
    e.r = tab.rank[e.s];
    e.EC = expand_cols(e.r);
    const int TGs = ceil_div_i(e.n, kTG);
    const int tg = l % TGs;
    l /= TGs;
    int i = 0;
    while (i < sh.n - 1) {
        const int nc = ceil_div_i(sh.off[i + 1] - sh.off[i], e.EC);
        if (l < nc) break;
        l -= nc;
        ++i;
    }
    e.i = i;
    e.c0 = l * e.EC;
    e.EW = min(e.EC, sh.off[i + 1] - sh.off[i] - e.c0);
    e.tok0 = tg * kTG;
    e.ntok = min(kTG, e.n - e.tok0);
    return e;
}

__device__ __forceinline__ int shrink_units_of(int n, int r, const Shape &sh) {
    return sh.n * ceil_div_i(r, kRG) * ceil_div_i(n, kTG) * ceil_div_i(sh.k, kKC);
}

__device__ __forceinline__ int expand_units_of(int n, int r, const Shape &sh) {
    const int ec = expand_cols(r);
    int c = 0;
    for (int i = 0; i < sh.n; ++i) c += ceil_div_i(sh.off[i + 1] - sh.off[i], ec);
    return c * ceil_div_i(n, kTG);
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) fused_decode_kernel(Ctx c, Shape sh, const void *__restrict__ table) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;                                                  // kStages x kStageBytes
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + kStages * kStageBytes);  // [kStages]
    uint64_t *empty = full + kStages;                                            // [kStages]
    uint64_t *cbar = empty + kStages;                                            // [1] consumer barrier
    float *scratch = reinterpret_cast<float *>(cbar + 2);                        // [kCWarps][8 x 16]
    int32_t *pref_s = reinterpret_cast<int32_t *>(scratch + kCWarps * 128);     // [S]
    int32_t *pref_e = pref_s + sh.S;                                             // [S]
    int32_t *scan_scr = pref_e + sh.S;                                           // [33]
    volatile int32_t *abort_flag = scan_scr + 33;                                // [1]
    volatile int32_t *ready_flag = scan_scr + 34;                                // [kStages]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
    const TableView tab(table, sh.S, sh.n);

    // Prologue: work units per slot, identical in every CTA.
    const int32_t *hdr = static_cast<const int32_t *>(table);
    const bool ok = hdr[0] == kTableMagic && hdr[1] == sh.S && hdr[2] == sh.n && c.seg[sh.S + 1] == c.T;
    if (!ok && tid == 0 && blockIdx.x == 0) report_error(c.err, LORA_ERR_INVALID_ARG);
    for (int s = tid; s < sh.S; s += blockDim.x) {
        const int n = ok ? c.seg[s + 1] - c.seg[s] : 0;
        const int r = ok ? tab.rank[s] : 0;
        const bool rank_ok = r <= sh.r_max;
        if (!rank_ok && blockIdx.x == 0) report_error(c.err, LORA_ERR_RANK);
        const bool act = ok && rank_ok && n > 0 && r > 0;
        pref_s[s] = act ? shrink_units_of(n, r, sh) : 0;
        pref_e[s] = act ? expand_units_of(n, r, sh) : 0;
    }
    if (tid == 0) {
        *abort_flag = 0;
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kCWarps);
        }
        mbar_init(cbar, kCWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int32_t NS = block_exclusive_scan(pref_s, sh.S, scan_scr);
    const int32_t NE = block_exclusive_scan(pref_e, sh.S, scan_scr);
    const int32_t G = gridDim.x, b = blockIdx.x;
    // this CTA's units: shrink b, b+G, ..., then expand b, b+G, ...
    const int32_t my_s = NS > b ? ceil_div_i(NS - b, G) : 0;
    const int32_t my_e = NE > b ? ceil_div_i(NE - b, G) : 0;
    const int32_t my_total = my_s + my_e;

    if (warp == kCWarps) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t parity = 1;  // first pass over the ring does not wait
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
                const ShrinkUnit w = decode_shrink(b + it * G, pref_s, sh, tab, c.seg);
                const uint32_t row_bytes = static_cast<uint32_t>(w.W) * 2u;
                if (lane == 0) mbar_arrive_expect_tx(&full[stage], row_bytes * static_cast<uint32_t>(w.R + w.ntok));
                __syncwarp();
                const uint16_t *A = reinterpret_cast<const uint16_t *>(tab.a_ptr[w.s * sh.n + w.i]);
                for (int j = lane; j < w.R + w.ntok; j += 32) {
                    if (j < w.R) {
                        const uint16_t *src = A + static_cast<int64_t>(w.rg * kRG + j) * sh.k + w.kc0;
                        bulk_g2s(st + j * kPitch, src, row_bytes, &full[stage]);
                    } else {
                        const int tt = j - w.R;
                        const int32_t t = c.sorted_ids[w.p0 + w.tok0 + tt];
                        const uint16_t *src = c.x + static_cast<int64_t>(t) * c.ldx + w.kc0;
                        bulk_g2s(st + (kRG + tt) * kPitch, src, row_bytes, &full[stage]);
                    }
                }
            } else {
                const ExpandUnit e = decode_expand(b + (it - my_s) * G, pref_e, sh, tab, c.seg);
                const uint32_t b_bytes = static_cast<uint32_t>(e.EW) * static_cast<uint32_t>(e.r) * 2u;
                const uint32_t y_bytes = static_cast<uint32_t>(e.EW) * 2u;
                const int ypitch = e.EC * 2 + 64;
                if (lane == 0) mbar_arrive_expect_tx(&full[stage], b_bytes + y_bytes * static_cast<uint32_t>(e.ntok));
                __syncwarp();
                if (lane == 0) {
                    const uint16_t *B = reinterpret_cast<const uint16_t *>(tab.b_ptr[e.s * sh.n + e.i]);
                    bulk_g2s(st, B + static_cast<int64_t>(e.c0) * e.r, b_bytes, &full[stage]);
                }
                for (int tt = lane; tt < e.ntok; tt += 32) {
                    const int32_t t = c.sorted_ids[e.p0 + e.tok0 + tt];
                    const uint16_t *src = c.y + static_cast<int64_t>(t) * c.ldy + sh.off[e.i] + e.c0;
                    bulk_g2s(st + kBTileBytes + tt * ypitch, src, y_bytes, &full[stage]);
                }
            }
            ++issued;
            if (++stage == kStages) {
                stage = 0;
                parity ^= 1u;
            }
        }
        // On abort, the copies already issued must land before the CTA exits:
        // wait (bounded) for the last phase of every stage that was filled.
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
    float *scr = scratch + warp * 128;
    int stage = 0;
    uint32_t parity = 0, cphase = 0;
    for (int32_t it = 0; it < my_total; ++it) {
        bool got = mbar_wait(&full[stage], parity, abort_flag);
        if (!got) {
            if (lane == 0) {
                *abort_flag = 1;
                report_error(c.err, LORA_ERR_TIMEOUT);
            }
            break;
        }
        const unsigned char *st = ring + stage * kStageBytes;
        if (it < my_s) {
            // ------------------------------------------------------- shrink unit
            const ShrinkUnit w = decode_shrink(b + it * G, pref_s, sh, tab, c.seg);
            const int nb = ceil_div_i(w.R, 16), ntt = ceil_div_i(w.ntok, 8), kblocks = ceil_div_i(w.W, 32);
            const unsigned char *sA = st, *sX = st + kRG * kPitch;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int tile = warp; tile < nb * ntt; tile += kCWarps) {
                const int rb = tile % nb, tt = tile / nb;
                const int ra = rb * 16 + g, rb2 = ra + 8, tk = tt * 8 + g;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int kb = 0; kb < kblocks; ++kb) {
                    const int col = kb * 32 + 8 * q;
                    const bool cok = col < w.W;
                    const uint4 va = (cok && ra < w.R) ? lds128(sA + ra * kPitch + col * 2) : z;
                    const uint4 vb = (cok && rb2 < w.R) ? lds128(sA + rb2 * kPitch + col * 2) : z;
                    const uint4 xv = (cok && tk < w.ntok) ? lds128(sX + tk * kPitch + col * 2) : z;
                    mma_bf16_16816(acc, va.x, vb.x, va.y, vb.y, xv.x, xv.y);
                    mma_bf16_16816(acc, va.z, vb.z, va.w, vb.w, xv.z, xv.w);
                }
                // transpose to [token][rank] through the warp's scratch, then add 4 ranks at a time
                scr[(2 * q) * 16 + g] = acc[0];
                scr[(2 * q + 1) * 16 + g] = acc[1];
                scr[(2 * q) * 16 + g + 8] = acc[2];
                scr[(2 * q + 1) * 16 + g + 8] = acc[3];
                __syncwarp();
                const int tl = lane >> 2, jq = lane & 3;
                if (tt * 8 + tl < w.ntok && rb * 16 + 4 * jq < w.R) {
                    const float4 v = *reinterpret_cast<const float4 *>(scr + tl * 16 + 4 * jq);
                    const int32_t t = c.sorted_ids[w.p0 + w.tok0 + tt * 8 + tl];
                    float *dst = c.acc + (static_cast<int64_t>(w.i) * c.T + t) * sh.r_max + w.rg * kRG + rb * 16 + 4 * jq;
                    red_add_v4(dst, v.x, v.y, v.z, v.w);
                }
                __syncwarp();
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[stage]);
                atomicAdd(&c.shrink_done[w.s * LORA_MAX_SLICES + w.i], 1);
            }
        } else {
            // ------------------------------------------------------- expand unit
            const ExpandUnit e = decode_expand(b + (it - my_s) * G, pref_e, sh, tab, c.seg);
            const int nt8 = e.EW / 8, npairs = ceil_div_i(nt8, 2), ntt = ceil_div_i(e.ntok, 16);
            const int ypitch = e.EC * 2 + 64;
            const int ctr = e.s * LORA_MAX_SLICES + e.i;
            const int64_t acc_slice = static_cast<int64_t>(e.i) * c.T;
            // wait until every shrink unit of this (slot, slice) has been added
            const int32_t need = kCWarps * ceil_div_i(e.r, kRG) * ceil_div_i(e.n, kTG) * ceil_div_i(sh.k, kKC);
            if (warp == 0 && lane == 0) {
                int32_t ready = 1;
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire(&c.shrink_done[ctr]) < need) {
                    if (globaltimer_ns() - t0 > kWaitNs) {
                        ready = 0;
                        report_error(c.err, LORA_ERR_TIMEOUT);
                        break;
                    }
                }
                ready_flag[stage] = ready;
            }
            if (!consumer_barrier(cbar, cphase, abort_flag)) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report_error(c.err, LORA_ERR_TIMEOUT);
                }
                break;
            }
            const bool ready = ready_flag[stage] != 0;
            // stage the unit's accumulator rows once, as bf16 hi and lo parts
            // (xa = hi + lo to about 2^-17 relative)
            const bool staged = e.r <= kAccStageMaxR;
            const int apitch = frag_pitch(e.r);
            unsigned char *sHi = const_cast<unsigned char *>(st) + kAccOff;
            unsigned char *sLo = sHi + kTG * apitch;
            if (staged) {
                const int r4 = ready ? e.r / 4 : 0;
                for (int idx = tid; idx < e.ntok * r4; idx += kCWarps * 32) {
                    const int row = idx / r4, j4 = idx % r4;
                    const int32_t t = c.sorted_ids[e.p0 + e.tok0 + row];
                    const float4 v = ldg_cg_f4(c.acc + (acc_slice + t) * sh.r_max + 4 * j4);
                    uint32_t h0, l0, h1, l1;
                    split_bf16x2(v.x, v.y, h0, l0);
                    split_bf16x2(v.z, v.w, h1, l1);
                    sts64(sHi + row * apitch + j4 * 8, h0, h1);
                    sts64(sLo + row * apitch + j4 * 8, l0, l1);
                }
                if (!consumer_barrier(cbar, cphase, abort_flag)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report_error(c.err, LORA_ERR_TIMEOUT);
                    }
                    break;
                }
            }
            const unsigned char *sB = st, *sY = st + kBTileBytes;
            const float scale = tab.scale[e.s];
            const int kbn = ceil_div_i(e.r, 32);
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int item = warp; ready && item < ntt * npairs; item += kCWarps) {
                const int tt = item / npairs, pair = item % npairs;
                const int ra = tt * 16 + g, rb2 = ra + 8;
                const int32_t ta = ra < e.ntok ? c.sorted_ids[e.p0 + e.tok0 + ra] : -1;
                const int32_t tb = rb2 < e.ntok ? c.sorted_ids[e.p0 + e.tok0 + rb2] : -1;
                float acc[2][4];
#pragma unroll
                for (int u = 0; u < 2; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
                for (int kb = 0; kb < kbn; ++kb) {
                    const int j = kb * 32 + 8 * q;
                    const bool jok = j < e.r;
                    uint4 ha, la, hb, lb;  // A operand rows g (token ta) and g+8 (token tb)
                    if (staged) {
                        ha = (jok && ta >= 0) ? lds128(sHi + ra * apitch + j * 2) : z;
                        la = (jok && ta >= 0) ? lds128(sLo + ra * apitch + j * 2) : z;
                        hb = (jok && tb >= 0) ? lds128(sHi + rb2 * apitch + j * 2) : z;
                        lb = (jok && tb >= 0) ? lds128(sLo + rb2 * apitch + j * 2) : z;
                    } else {
                        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
                        if (jok && ta >= 0) {
                            const float *p = c.acc + (acc_slice + ta) * sh.r_max + j;
                            a0 = ldg_cg_f4(p);
                            a1 = ldg_cg_f4(p + 4);
                        }
                        if (jok && tb >= 0) {
                            const float *p = c.acc + (acc_slice + tb) * sh.r_max + j;
                            b0 = ldg_cg_f4(p);
                            b1 = ldg_cg_f4(p + 4);
                        }
                        split_bf16x2(a0.x, a0.y, ha.x, la.x);
                        split_bf16x2(a0.z, a0.w, ha.y, la.y);
                        split_bf16x2(a1.x, a1.y, ha.z, la.z);
                        split_bf16x2(a1.z, a1.w, ha.w, la.w);
                        split_bf16x2(b0.x, b0.y, hb.x, lb.x);
                        split_bf16x2(b0.z, b0.w, hb.y, lb.y);
                        split_bf16x2(b1.x, b1.y, hb.z, lb.z);
                        split_bf16x2(b1.z, b1.w, hb.w, lb.w);
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = pair * 16 + 4 * (g >> 1) + 2 * u + (g & 1);
                        const uint4 bv = (jok && col < e.EW) ? lds128(sB + (col * e.r + j) * 2) : z;
                        mma_bf16_16816(acc[u], ha.x, hb.x, ha.y, hb.y, bv.x, bv.y);
                        mma_bf16_16816(acc[u], ha.z, hb.z, ha.w, hb.w, bv.z, bv.w);
                        mma_bf16_16816(acc[u], la.x, lb.x, la.y, lb.y, bv.x, bv.y);
                        mma_bf16_16816(acc[u], la.z, lb.z, la.w, lb.w, bv.z, bv.w);
                    }
                }
                // y = y + scale * acc, one rounding; lane owns 4 consecutive columns
                const int col0 = pair * 16 + 4 * q;
                if (col0 < e.EW) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int32_t t = half == 0 ? ta : tb;
                        const int row = half == 0 ? ra : rb2;
                        if (t < 0) continue;
                        const uint2 yv = lds64(sY + row * ypitch + col0 * 2);
                        const float v0 = fmaf(scale, acc[0][2 * half + 0], bf16lo_to_f32(yv.x));
                        const float v1 = fmaf(scale, acc[0][2 * half + 1], bf16hi_to_f32(yv.x));
                        const float v2 = fmaf(scale, acc[1][2 * half + 0], bf16lo_to_f32(yv.y));
                        const float v3 = fmaf(scale, acc[1][2 * half + 1], bf16hi_to_f32(yv.y));
                        stg_u2(c.y + static_cast<int64_t>(t) * c.ldy + sh.off[e.i] + e.c0 + col0, pack_bf16x2(v0, v1),
                               pack_bf16x2(v2, v3));
                    }
                }
            }
            __threadfence();
            __syncwarp();
            int32_t old = 0;
            if (lane == 0) {
                mbar_arrive(&empty[stage]);
                old = atom_add_acq_rel(&c.expand_done[ctr], 1);
            }
            old = __shfl_sync(0xffffffffu, old, 0);
            // expand warps of this (slot, slice): kCWarps per unit, units = column chunks x token groups
            const int32_t e_need = kCWarps * ceil_div_i(sh.off[e.i + 1] - sh.off[e.i], e.EC) * ceil_div_i(e.n, kTG);
            if (old == e_need - 1) {
                // last reader of this (slot, slice): clear its accumulator rows and the counters
                const int r4 = e.r / 4;
                for (int idx = lane; idx < e.n * r4; idx += 32) {
                    const int tk = idx / r4, j4 = idx % r4;
                    const int32_t t = c.sorted_ids[e.p0 + tk];
                    *reinterpret_cast<float4 *>(c.acc + (acc_slice + t) * sh.r_max + 4 * j4) =
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

size_t fused_smem_bytes(int32_t S) {
    return size_t(kStages) * kStageBytes + (2 * kStages + 2) * sizeof(uint64_t) + kCWarps * 128 * sizeof(float) +
           sizeof(int32_t) * (2 * size_t(S) + 40);
}

}  // namespace

bool fused_decode_available() { return false; }

cudaError_t launch_fused_decode(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                const void *table, const int32_t *sorted_ids, const int32_t *seg, float *ws,
                                int32_t T, int32_t *err, cudaStream_t stream) {
    static int num_sms = 0;
    static bool attr_set = false;
    if (!attr_set) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(fused_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(fused_smem_bytes(LORA_MAX_SLOTS)));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_decode_kernel, kThreads,
                                                          fused_smem_bytes(LORA_MAX_SLOTS));
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        attr_set = true;
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
    cfg.dynamicSmemBytes = fused_smem_bytes(sh.S);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_decode_kernel, c, sh, table);
}

}  // namespace lora
