// Decode-size LoRA branch: shrink and expand kernels on warp-level tensor-core MMA.
//
// Shrink (vLLM book ch. 16, section 16.4.2, lora_shrink: buffer[t, :] = x[t, :] A_slot)
// computes xa[i][t][0..r_s) for every token t of an active slot s.  One work item
// is (slot, slice, 64 rank rows, 64 tokens); it is split over k across the CTAs
// of a thread-block cluster (split-K: M = tokens is small and K = k is large,
// TensorRT-LLM LoRA serving page, "path 2: split-K tuning").  Each CTA reduces
// its warps' partials in shared memory, then the cluster reduces the CTA
// partials through distributed shared memory in a fixed order and writes xa
// once: deterministic, no atomics and no zeroed buffer.
//
// Expand (same book section, lora_expand: out[t, slice] += buffer[t, :] B_slot)
// computes y[t, o_i + m] += scale_s * sum_j xa[i][t][j] B_s,i[m, j].  One work item
// is (slot, slice, 512 output columns); each warp owns 64 columns, keeps their B
// rows in registers and sweeps all tokens of the slot 16 at a time, reading and
// writing y with 16-byte accesses.  Launched as a programmatic dependent of the
// shrink, it loads B before waiting for the shrink grid.
//
// Both use mma.sync m16n8k16 (bf16 in, fp32 accumulate).  Because the reduction
// over k (or j) is order-free, each lane loads 8 consecutive bf16 (16 bytes) of
// a row and feeds them to two MMAs: logical k {2q, 2q+1, 2q+8, 2q+9} of the
// first MMA are physical offsets {0, 1, 2, 3} of the lane's 8, those of the
// second MMA are {4, 5, 6, 7}.  The same permutation is used for both operands,
// so every load is a 128-bit vector load of contiguous memory.
#include <algorithm>

#include "common.cuh"

namespace lora {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kShrTok = 64;    // tokens per shrink item: 8 MMA n-tiles of 8
constexpr int kShrRows = 64;   // rank rows per shrink item: 4 MMA m-blocks of 16
constexpr int kExpCols = 512;  // output columns per expand item: 8 warps x 64

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Activations: read-only for the kernel, shared by several warps of a CTA, so
// they may stay in L1.
__device__ __forceinline__ uint4 ldg_act(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// Shrink
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) shrink_kernel(
    const uint16_t *__restrict__ x, int64_t ldx, Shape sh, const void *__restrict__ table,
    const int32_t *__restrict__ sorted_ids, const int32_t *__restrict__ seg, float *__restrict__ xa,
    int32_t T, int32_t *err, int32_t trigger_dependents) {
    extern __shared__ __align__(16) unsigned char smem[];
    float *s_red = reinterpret_cast<float *>(smem);                                // [8 warps][16][64 tok]
    float *s_part = s_red + kWarps * 16 * kShrTok;                                 // [64 tok][64 rows]
    int32_t *s_pref = reinterpret_cast<int32_t *>(s_part + kShrTok * kShrRows);    // [S]
    int32_t *s_scr = s_pref + sh.S;                                                // [33]

    if (trigger_dependents) pdl_launch_dependents();
    const uint32_t KS = cluster_nctarank(), crank = cluster_ctarank();
    const int32_t cid = static_cast<int32_t>(blockIdx.x / KS);
    const TableView tab(table, sh.S, sh.n);
    const int32_t n_sl = sh.n;
    const int32_t total = slot_item_prefix(table, sh, seg, T, s_pref, s_scr, err, [&](int32_t n, int32_t r) {
        return n_sl * ((r + kShrRows - 1) / kShrRows) * ((n + kShrTok - 1) / kShrTok);
    });
    if (cid >= total) return;  // the same for every CTA of the cluster

    const int32_t s = find_slot(s_pref, sh.S, cid);
    int32_t l = cid - s_pref[s];
    const int32_t p0 = seg[s], n_s = seg[s + 1] - p0, r = tab.rank[s];
    const int32_t RG = (r + kShrRows - 1) / kShrRows, TG = (n_s + kShrTok - 1) / kShrTok;
    const int32_t tg = l % TG;
    l /= TG;
    const int32_t rg = l % RG;
    const int32_t i = l / RG;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, q = lane & 3;
    const int32_t row0 = rg * kShrRows;
    const int32_t R = min(kShrRows, r - row0);      // multiple of 8
    const int32_t nb = (R + 15) >> 4;               // 16-row m-blocks in use
    const int32_t wsub = kWarps / nb;               // warps sharing one m-block (split k)
    const int32_t rb = warp % nb, sub = warp / nb;
    const int32_t tok0 = tg * kShrTok;
    const int32_t ntok = min(kShrTok, n_s - tok0);
    const int32_t ntiles = (ntok + 7) >> 3;
    const int32_t k = sh.k;
    const int32_t KB = (k + 31) >> 5;               // 32-wide k blocks
    const int32_t kb_lo = static_cast<int32_t>(crank * KB / KS);
    const int32_t kb_hi = static_cast<int32_t>((crank + 1) * KB / KS);

    float acc[8][4];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;

    if (sub < wsub) {
        const int32_t len = kb_hi - kb_lo;
        const int32_t wb_lo = kb_lo + sub * len / wsub, wb_hi = kb_lo + (sub + 1) * len / wsub;
        const uint16_t *A = reinterpret_cast<const uint16_t *>(tab.a_ptr[s * n_sl + i]);
        const int32_t j_lo = row0 + rb * 16 + g, j_hi = j_lo + 8;
        const bool lo_ok = j_lo < r, hi_ok = j_hi < r;
        const uint16_t *a_lo = A + static_cast<int64_t>(lo_ok ? j_lo : 0) * k + 8 * q;
        const uint16_t *a_hi = A + static_cast<int64_t>(hi_ok ? j_hi : 0) * k + 8 * q;
        const uint16_t *xr[8];
        bool xok[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            xok[u] = (8 * u + g) < ntok;
            const int32_t t = xok[u] ? sorted_ids[p0 + tok0 + 8 * u + g] : 0;
            xr[u] = x + static_cast<int64_t>(t) * ldx + 8 * q;
        }
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 2
        for (int32_t kb = wb_lo; kb < wb_hi; ++kb) {
            const int32_t c = kb * 32;
            const bool cok = c + 8 * q < k;
            const uint4 va = (lo_ok && cok) ? ldg_stream(a_lo + c) : z;
            const uint4 vb = (hi_ok && cok) ? ldg_stream(a_hi + c) : z;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (u < ntiles) {
                    const uint4 xv = (xok[u] && cok) ? ldg_act(xr[u] + c) : z;
                    mma_bf16_16816(acc[u], va.x, vb.x, va.y, vb.y, xv.x, xv.y);
                    mma_bf16_16816(acc[u], va.z, vb.z, va.w, vb.w, xv.z, xv.w);
                }
            }
        }
        // warp partial -> s_red[warp][row][tok]
        float *red = s_red + warp * 16 * kShrTok;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            red[g * kShrTok + 8 * u + 2 * q] = acc[u][0];
            red[g * kShrTok + 8 * u + 2 * q + 1] = acc[u][1];
            red[(g + 8) * kShrTok + 8 * u + 2 * q] = acc[u][2];
            red[(g + 8) * kShrTok + 8 * u + 2 * q + 1] = acc[u][3];
        }
    }
    __syncthreads();
    // CTA partial: sum the warps that split k for each m-block, in warp order
    for (int e = threadIdx.x; e < nb * 16 * kShrTok; e += kThreads) {
        const int row = e / kShrTok, tok = e % kShrTok;
        const int rbx = row >> 4, rr = row & 15;
        float v = 0.f;
        for (int sb = 0; sb < wsub; ++sb) v += s_red[(rbx + nb * sb) * 16 * kShrTok + rr * kShrTok + tok];
        s_part[tok * kShrRows + row] = v;
    }
    cluster_sync();
    // Cluster reduction: CTA c owns an equal share of the (token, 4-row) outputs
    // and sums that share over all CTAs of the cluster in rank order.
    const int32_t RQ = R >> 2;
    const int32_t nq = ntok * RQ;
    const int32_t e_lo = static_cast<int32_t>(crank * nq / KS), e_hi = static_cast<int32_t>((crank + 1) * nq / KS);
    const uint32_t base = smem_addr(s_part);
    for (int32_t e = e_lo + threadIdx.x; e < e_hi; e += kThreads) {
        const int32_t tok = e / RQ, rq = e % RQ;
        const uint32_t off = static_cast<uint32_t>((tok * kShrRows + 4 * rq) * sizeof(float));
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (uint32_t c = 0; c < KS; ++c) {
            const float4 w = ld_dsmem_f4(map_to_rank(base + off, c));
            v.x += w.x;
            v.y += w.y;
            v.z += w.z;
            v.w += w.w;
        }
        const int32_t t = sorted_ids[p0 + tok0 + tok];
        *reinterpret_cast<float4 *>(xa + (static_cast<int64_t>(i) * T + t) * sh.r_max + row0 + 4 * rq) = v;
    }
    cluster_sync();  // keep this CTA's shared memory alive until the cluster has read it
}

// ---------------------------------------------------------------------------
// Expand
// ---------------------------------------------------------------------------
struct ExpandArgs {
    const float *xa;
    uint16_t *y;
    int64_t ldy;
    int32_t T;
    int32_t *err;
};

// Columns owned by lane (g, q) in n-tile u of a warp's 64 columns: the D fragment
// gives the lane logical columns 2q, 2q+1 of each n-tile; they are placed at
// physical columns 16q + 2u + {0, 1}, so a lane owns 16 consecutive columns of
// y.  The B operand row a lane loads for n-tile u is column 16(g/2) + 2u + g%2.
__device__ __forceinline__ int32_t b_col(int g, int u) { return 16 * (g >> 1) + 2 * u + (g & 1); }

__global__ void __launch_bounds__(kThreads) expand_kernel(
    ExpandArgs a, Shape sh, const void *__restrict__ table, const int32_t *__restrict__ sorted_ids,
    const int32_t *__restrict__ seg, int32_t wait_primary) {
    extern __shared__ __align__(16) unsigned char smem[];
    int32_t *s_pref = reinterpret_cast<int32_t *>(smem);
    int32_t *s_scr = s_pref + sh.S;

    const TableView tab(table, sh.S, sh.n);
    int32_t chunks[LORA_MAX_SLICES];
    int32_t chunks_total = 0;
#pragma unroll
    for (int i = 0; i < LORA_MAX_SLICES; ++i) {
        chunks[i] = i < sh.n ? (sh.off[i + 1] - sh.off[i] + kExpCols - 1) / kExpCols : 0;
        chunks_total += chunks[i];
    }
    const int32_t total = slot_item_prefix(table, sh, seg, a.T, s_pref, s_scr, a.err,
                                           [&](int32_t, int32_t) { return chunks_total; });
    if (static_cast<int32_t>(blockIdx.x) >= total) return;
    const int32_t s = find_slot(s_pref, sh.S, blockIdx.x);
    int32_t l = blockIdx.x - s_pref[s];
    int32_t i = 0;
    while (l >= chunks[i]) {
        l -= chunks[i];
        ++i;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, q = lane & 3;
    const int32_t d_i = sh.off[i + 1] - sh.off[i];
    const int32_t c0 = l * kExpCols + warp * 64;
    if (c0 >= d_i) return;  // no block-level barrier below this point
    const int32_t p0 = seg[s], n_s = seg[s + 1] - p0, r = tab.rank[s];
    const float scale = tab.scale[s];
    const uint16_t *B = reinterpret_cast<const uint16_t *>(tab.b_ptr[s * sh.n + i]);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);

    uint4 bf[2][8];
    auto load_b = [&](int32_t rc) {
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int32_t col = c0 + b_col(g, u);
                const int32_t j = rc + 32 * kb + 8 * q;
                bf[kb][u] = (col < d_i && j < r) ? ldg_stream(B + static_cast<int64_t>(col) * r + j) : z;
            }
        }
    };
    if (r <= 64) load_b(0);
    if (wait_primary) pdl_wait();

    const int64_t xa_slice = static_cast<int64_t>(i) * a.T;
    const int32_t ntt = (n_s + 15) >> 4;
    for (int32_t tt = 0; tt < ntt; ++tt) {
        const int32_t pa = tt * 16 + g, pb = pa + 8;
        const int32_t ta = pa < n_s ? sorted_ids[p0 + pa] : -1;
        const int32_t tb = pb < n_s ? sorted_ids[p0 + pb] : -1;
        float acc[8][4];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
        for (int32_t rc = 0; rc < r; rc += 64) {
            if (r > 64) load_b(rc);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                if (rc + 32 * kb < r) {
                    const int32_t j = rc + 32 * kb + 8 * q;
                    float4 ea0 = make_float4(0.f, 0.f, 0.f, 0.f), ea1 = ea0, eb0 = ea0, eb1 = ea0;
                    if (ta >= 0 && j < r) {
                        const float *p = a.xa + (xa_slice + ta) * sh.r_max + j;
                        ea0 = ldg_cg_f4(p);
                        ea1 = ldg_cg_f4(p + 4);
                    }
                    if (tb >= 0 && j < r) {
                        const float *p = a.xa + (xa_slice + tb) * sh.r_max + j;
                        eb0 = ldg_cg_f4(p);
                        eb1 = ldg_cg_f4(p + 4);
                    }
                    // A operand rows: g <- token ta, g+8 <- token tb
                    uint32_t h0, l0, h1, l1, h2, l2, h3, l3, h4, l4, h5, l5, h6, l6, h7, l7;
                    split_bf16x2(ea0.x, ea0.y, h0, l0);  // row g,   k-half 0, logical 2q..2q+1
                    split_bf16x2(eb0.x, eb0.y, h1, l1);  // row g+8, k-half 0
                    split_bf16x2(ea0.z, ea0.w, h2, l2);  // row g,   k-half 0, logical 2q+8..
                    split_bf16x2(eb0.z, eb0.w, h3, l3);  // row g+8
                    split_bf16x2(ea1.x, ea1.y, h4, l4);  // k-half 1
                    split_bf16x2(eb1.x, eb1.y, h5, l5);
                    split_bf16x2(ea1.z, ea1.w, h6, l6);
                    split_bf16x2(eb1.z, eb1.w, h7, l7);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint4 bv = bf[kb][u];
                        mma_bf16_16816(acc[u], h0, h1, h2, h3, bv.x, bv.y);
                        mma_bf16_16816(acc[u], h4, h5, h6, h7, bv.z, bv.w);
                        mma_bf16_16816(acc[u], l0, l1, l2, l3, bv.x, bv.y);
                        mma_bf16_16816(acc[u], l4, l5, l6, l7, bv.z, bv.w);
                    }
                }
            }
        }
        // y read-modify-write: lane owns columns c0 + 16q + [0, 16) of rows ta and tb
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int32_t t = half == 0 ? ta : tb;
            if (t < 0) continue;
            uint16_t *yr = a.y + static_cast<int64_t>(t) * a.ldy + sh.off[i] + c0 + 16 * q;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (c0 + 16 * q + 8 * h < d_i) {
                    uint4 yv = *reinterpret_cast<const uint4 *>(yr + 8 * h);
                    uint32_t w[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                    for (int m2 = 0; m2 < 4; ++m2) {
                        const int u = 4 * h + m2;
                        const float lo = fmaf(scale, acc[u][2 * half + 0], bf16lo_to_f32(w[m2]));
                        const float hi = fmaf(scale, acc[u][2 * half + 1], bf16hi_to_f32(w[m2]));
                        w[m2] = pack_bf16x2(lo, hi);
                    }
                    stg_u4(yr + 8 * h, make_uint4(w[0], w[1], w[2], w[3]));
                }
            }
        }
    }
}

__global__ void premultiply_kernel(uint16_t *w, int64_t n, float scale) {
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < n; e += int64_t(gridDim.x) * blockDim.x) {
        const float v = __uint_as_float(static_cast<uint32_t>(w[e]) << 16) * scale;
        w[e] = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xffffu);
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Host-side launchers
// ---------------------------------------------------------------------------
static size_t shrink_smem(int32_t S) {
    return sizeof(float) * (kWarps * 16 * kShrTok + kShrTok * kShrRows) + sizeof(int32_t) * (size_t(S) + 40);
}

static size_t expand_smem(int32_t S) { return sizeof(int32_t) * (size_t(S) + 40); }

static int shrink_cluster_size(int32_t k) {
    int ks = k / 512;  // about 512 columns of k per CTA
    if (ks < 1) ks = 1;
    if (ks > 8) ks = 8;
    return ks;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

cudaError_t launch_shrink(const uint16_t *x, int64_t ldx, const Shape &sh, const void *table,
                          const int32_t *sorted_ids, const int32_t *seg, float *xa, int32_t T, int32_t *err,
                          bool trigger_dependents, cudaStream_t stream) {
    const size_t smem = shrink_smem(sh.S);
    // per call: the attribute belongs to the current device's context
    cudaError_t ea = cudaFuncSetAttribute(shrink_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (ea != cudaSuccess) return ea;
    const int ks = shrink_cluster_size(sh.k);
    // upper bound on items: slices x rank groups x token groups (sum over slots
    // of ceil(n_s / 64) <= min(S, T) + T / 64)
    const int64_t tok_groups = std::min<int64_t>(sh.S, T) + ceil_div(T, kShrTok);
    const int64_t items = int64_t(sh.n) * ceil_div(sh.r_max, kShrRows) * tok_groups;
    if (items <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(items * ks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, shrink_kernel, reinterpret_cast<const uint16_t *>(x), ldx, sh, table,
                              sorted_ids, seg, xa, T, err, int32_t(trigger_dependents ? 1 : 0));
}

cudaError_t launch_expand(const float *xa, uint16_t *y, int64_t ldy, const Shape &sh, const void *table,
                          const int32_t *sorted_ids, const int32_t *seg, int32_t T, int32_t *err,
                          bool programmatic, cudaStream_t stream) {
    int64_t chunks = 0;
    for (int i = 0; i < sh.n; ++i) chunks += ceil_div(sh.off[i + 1] - sh.off[i], kExpCols);
    const int64_t items = std::min<int64_t>(sh.S, T) * chunks;
    if (items <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(items));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = expand_smem(sh.S);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    ExpandArgs a{xa, y, ldy, T, err};
    return cudaLaunchKernelEx(&cfg, expand_kernel, a, sh, table, sorted_ids, seg, int32_t(programmatic ? 1 : 0));
}

cudaError_t launch_premultiply(uint16_t *w, int64_t n, float scale, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>(ceil_div(n, 256), 4096);
    premultiply_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w, n, scale);
    return cudaGetLastError();
}

}  // namespace lora
