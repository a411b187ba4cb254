// Small-batch decode in one launch: one thread-block cluster per adapter slot.
//
// The branch of a slot s with tokens t (S-LoRA "Unified Paging and
// Heterogeneous Batching", the shrink and expand of a multi-adapter batch):
//     y[t, o_i + m] += scale_s * sum_j (sum_c x[t, c] A_{s,i}[j, c]) B_{s,i}[m, j].
// With few tokens per slot the call moves a few megabytes and is bound by the
// latency of its dependent steps.  This kernel keeps every step of a slot inside
// one cluster of KS = 16 CTAs (a cluster size above the portable 8, which this
// GPU allows):
//   - CTA c reads A_{s,i} rows over its share of k and the slot's x rows for
//     that share, and computes partial sums with warp MMAs (m16n8k16, bf16 in,
//     fp32 out);
//   - the KS partials meet through distributed shared memory: CTA c adds the
//     KS values of its share of the (token, rank) sums in rank order and writes
//     them, split into bf16 hi + lo parts, into the shared memory of every CTA;
//   - CTA c then applies B_{s,i} for its share of the output columns of every
//     slice, y read and written once, each value rounded once.
// The kernel is a programmatic dependent of the kernel before it on the stream:
// the slot table, the index (segment offsets and token ids) and the A and B rows
// are read before griddepcontrol.wait, x and y after it, so the only round
// trips after the wait are the x and y copies and two cluster barriers.  Tokens
// are taken 16 at a time (one MMA row block); a slot with more loops over its
// chunks.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "tc.cuh"

namespace lora {
namespace {

constexpr int kCThreads = 256;             // 8 warps
constexpr int kCTok = 16;                  // tokens per chunk: one MMA row block
constexpr int kCSmemLimit = 227 * 1024;

// Shared-memory layout of a CTA (byte offsets), the same on host and device.
struct CLayout {
    int32_t rp8, rp16, kcw, kcwp, ars, ncol, brs, srs, yrs;
    uint32_t a_off, x_off, p_off, s_off, b_off, y_off, tok_off, bytes;
};

// Output columns of slice i that each CTA takes: d_i / KS rounded up to 8.
__host__ __device__ inline int32_t slice_share(int32_t di, int32_t KS) { return ((di + KS - 1) / KS + 7) & ~7; }

__host__ __device__ inline CLayout c_layout(const Shape &sh, int32_t KS) {
    CLayout L;
    L.rp8 = (sh.r_max + 7) & ~7;
    L.rp16 = (sh.r_max + 15) & ~15;
    const int32_t nk8 = sh.k / 8;
    L.kcw = ((nk8 + KS - 1) / KS) * 8;  // the widest share of k
    L.kcwp = (L.kcw + 15) & ~15;        // padded to whole MMA k-steps (zeros)
    L.ars = L.kcwp + 8;                 // row stride (elements) of the A and x tiles
    int32_t ncol = 0;
    for (int i = 0; i < sh.n; ++i) ncol += slice_share(sh.off[i + 1] - sh.off[i], KS);
    L.ncol = ncol;
    L.brs = L.rp16 + 8;            // B tile: [ncol][rp16] (+8: bank spread)
    L.srs = sh.n * L.rp16 + 8;     // sums tiles: [16][n rp16]
    L.yrs = L.ncol + 8;            // y tile: [16][ncol]
    uint32_t o = 0;
    L.a_off = o;
    o += static_cast<uint32_t>(sh.n * L.rp8 * L.ars * 2);
    L.x_off = o;
    o += static_cast<uint32_t>(kCTok * L.ars * 2);
    L.p_off = o;
    o += static_cast<uint32_t>(kCTok * sh.n * L.rp8 * 4);
    L.s_off = o;
    o += static_cast<uint32_t>(2 * kCTok * L.srs * 2);
    L.b_off = o;
    o += static_cast<uint32_t>(L.ncol * L.brs * 2);
    L.y_off = o;
    o += static_cast<uint32_t>(kCTok * L.yrs * 2);
    L.tok_off = o;
    o += static_cast<uint32_t>(kCTok * 4);
    L.bytes = o;
    return L;
}

struct CArgs {
    const uint16_t *x;
    int64_t ldx;
    uint16_t *y;
    int64_t ldy;
    const void *table;
    const int32_t *sorted_ids;
    const int32_t *seg;
    int32_t *err;
    int32_t T;
    int32_t xdiv;  // x row of y row t: t / xdiv (routed experts sharing a token's x row)
};

__device__ __forceinline__ uint32_t lds32(const uint16_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_dsmem_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ uint16_t bf16_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

__global__ void __launch_bounds__(kCThreads) cluster_decode_kernel(const CArgs a, const Shape sh) {
    extern __shared__ __align__(16) unsigned char smem[];
    const uint32_t KS = cluster_nctarank(), c = cluster_ctarank();
    const CLayout L = c_layout(sh, static_cast<int32_t>(KS));
    const int32_t s = static_cast<int32_t>(blockIdx.y);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;

    // Every decision below that ends the CTA is the same in all CTAs of the
    // cluster (it reads the same table and index words), so no CTA leaves a
    // barrier that the others still wait at.  The table and the index are not
    // written by the kernel directly before this one (the index and plan
    // builders never start their dependents early), so they are read now.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int32_t *hdr = static_cast<const int32_t *>(a.table);
    if (!(hdr[0] == kTableMagic && hdr[1] == sh.S && hdr[2] == sh.n && a.seg[sh.S + 1] == a.T)) {
        if (s == 0 && c == 0 && tid == 0) report_error(a.err, LORA_ERR_INVALID_ARG);
        return;
    }
    const TableView tab(a.table, sh.S, sh.n);
    const int32_t r = tab.rank[s], p0 = a.seg[s], cnt = a.seg[s + 1] - p0;
    if (r > sh.r_max) {
        if (c == 0 && tid == 0) report_error(a.err, LORA_ERR_RANK);
        return;
    }
    if (r <= 0 || cnt <= 0 || p0 < 0 || p0 + cnt > a.T) return;
    const float scale = tab.scale[s];

    const uint32_t base = smem_addr(smem);
    const uint16_t *sX = reinterpret_cast<const uint16_t *>(smem + L.x_off);
    const uint16_t *sA = reinterpret_cast<const uint16_t *>(smem + L.a_off);
    const uint16_t *sB = reinterpret_cast<const uint16_t *>(smem + L.b_off);
    const uint16_t *sHi = reinterpret_cast<const uint16_t *>(smem + L.s_off);
    const uint16_t *sLo = sHi + kCTok * L.srs;
    float *sP = reinterpret_cast<float *>(smem + L.p_off);
    uint16_t *sY = reinterpret_cast<uint16_t *>(smem + L.y_off);
    int32_t *s_tok = reinterpret_cast<int32_t *>(smem + L.tok_off);

    // this CTA's share of k: 16-byte chunks [kc0, kc0 + kcw)
    const int32_t nk8 = sh.k / 8;
    const int32_t kc0 = static_cast<int32_t>(c * nk8 / KS) * 8;
    const int32_t kcw = static_cast<int32_t>((c + 1) * nk8 / KS) * 8 - kc0;
    const int32_t prs = sh.n * L.rp8;  // partial row: n slices of rp8 ranks

    // ---- A rows over the share of k (rows past r and columns past kcw: zeros) ----
    {
        const int32_t chunks = L.kcwp / 8;
        for (int32_t e = tid; e < prs * chunks; e += kCThreads) {
            const int32_t row = e / chunks, ch = e % chunks, i = row / L.rp8, j = row % L.rp8;
            const bool v = j < r && ch * 8 < kcw;
            const uint16_t *A = reinterpret_cast<const uint16_t *>(tab.a_ptr[s * sh.n + i]);
            tc::cp16(base + L.a_off + static_cast<uint32_t>((row * L.ars + ch * 8) * 2),
                     v ? A + static_cast<int64_t>(j) * sh.k + kc0 + ch * 8 : static_cast<const void *>(a.x), v);
        }
    }
    // ---- B rows of the CTA's output columns (ranks past r: zeros) ----
    {
        const int32_t chunks = L.rp16 / 8;
        int32_t colbase = 0;
        for (int i = 0; i < sh.n; ++i) {
            const int32_t di = sh.off[i + 1] - sh.off[i], dci = slice_share(di, static_cast<int32_t>(KS));
            const int32_t mc0 = static_cast<int32_t>(c) * dci, w = max(0, min(di, mc0 + dci) - mc0);
            const uint16_t *B = reinterpret_cast<const uint16_t *>(tab.b_ptr[s * sh.n + i]);
            if ((r & 7) == 0) {
                // rows of r ranks start on 16-byte boundaries
                for (int32_t e = tid; e < dci * chunks; e += kCThreads) {
                    const int32_t m = e / chunks, ch = e % chunks;
                    const bool v = m < w && ch * 8 < r;
                    tc::cp16(base + L.b_off + static_cast<uint32_t>(((colbase + m) * L.brs + ch * 8) * 2),
                             v ? B + static_cast<int64_t>(mc0 + m) * r + ch * 8 : static_cast<const void *>(a.x), v);
                }
            } else {
                uint16_t *dst = const_cast<uint16_t *>(sB);
                for (int32_t e = tid; e < dci * L.rp16; e += kCThreads) {
                    const int32_t m = e / L.rp16, j = e % L.rp16;
                    dst[(colbase + m) * L.brs + j] = (m < w && j < r) ? B[static_cast<int64_t>(mc0 + m) * r + j] : 0;
                }
            }
            colbase += dci;
        }
    }
    tc::cp_commit();
    // the sums tiles start at zero; ranks past r stay zero for every chunk
    for (int32_t e = tid; e < kCTok * L.srs; e += kCThreads)  // hi and lo: 2 x 16 x srs bf16 = 16 x srs words
        reinterpret_cast<uint32_t *>(smem + L.s_off)[e] = 0u;
    auto load_tokens = [&](int32_t chn) {
        const int32_t len = min(kCTok, cnt - chn * kCTok);
        if (tid < kCTok) {
            int32_t t = -1;
            if (tid < len) {
                t = a.sorted_ids[p0 + chn * kCTok + tid];
                if (t < 0 || t >= a.T) {
                    report_error(a.err, LORA_ERR_INVALID_ARG);
                    t = -1;
                }
            }
            s_tok[tid] = t;
        }
    };
    load_tokens(0);
    // x and y may be written by the kernel directly before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int32_t nchunks = (cnt + kCTok - 1) / kCTok;
    for (int32_t chn = 0; chn < nchunks; ++chn) {
        const int32_t len = min(kCTok, cnt - chn * kCTok);
        if (chn > 0) load_tokens(chn);
        for (int32_t e = tid; e < kCTok * prs; e += kCThreads) sP[e] = 0.f;
        __syncthreads();

        // ---- x rows of the chunk over the share of k, y rows over the CTA's columns ----
        {
            const int32_t chunks = L.kcwp / 8;
            for (int32_t e = tid; e < kCTok * chunks; e += kCThreads) {
                const int32_t row = e / chunks, ch = e % chunks, t = s_tok[row];
                const bool v = t >= 0 && ch * 8 < kcw;
                const int64_t xr = a.xdiv == 1 ? t : t / a.xdiv;
                tc::cp16(base + L.x_off + static_cast<uint32_t>((row * L.ars + ch * 8) * 2),
                         v ? a.x + xr * a.ldx + kc0 + ch * 8 : static_cast<const void *>(a.x), v);
            }
            int32_t colbase = 0;
            for (int i = 0; i < sh.n; ++i) {
                const int32_t di = sh.off[i + 1] - sh.off[i], dci = slice_share(di, static_cast<int32_t>(KS));
                const int32_t mc0 = static_cast<int32_t>(c) * dci, w = max(0, min(di, mc0 + dci) - mc0);
                const int32_t ych = dci / 8;
                for (int32_t e = tid; e < kCTok * ych; e += kCThreads) {
                    const int32_t row = e / ych, ch = e % ych, t = s_tok[row];
                    const bool v = t >= 0 && ch * 8 < w;
                    tc::cp16(base + L.y_off + static_cast<uint32_t>((row * L.yrs + colbase + ch * 8) * 2),
                             v ? a.y + static_cast<int64_t>(t) * a.ldy + sh.off[i] + mc0 + ch * 8
                               : static_cast<const void *>(a.y),
                             v);
                }
                colbase += dci;
            }
        }
        tc::cp_commit();
        tc::cp_wait_all();
        __syncthreads();

        // ---- shrink: partial[t][i rp8 + j] over the share of k; 8-rank column
        // blocks, split along k over the warps when there are fewer than 8 ----
        {
            const int32_t ncb = prs / 8, ksteps = L.kcwp / 16;
            const int32_t kq = max(1, 8 / ncb), items = ncb * kq;
            for (int32_t it = warp; it < items; it += kCThreads / 32) {
                const int32_t cb = it / kq, part = it % kq;
                if ((cb * 8) % L.rp8 >= r) continue;  // ranks past r: the partial stays zero
                const int32_t k_lo = part * ksteps / kq, k_hi = (part + 1) * ksteps / kq;
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                for (int32_t ks = k_lo; ks < k_hi; ++ks) {
                    const int32_t kk = ks * 16 + 2 * q;
                    const uint16_t *x0 = sX + g * L.ars + kk, *x1 = x0 + 8 * L.ars;
                    const uint16_t *ar = sA + (cb * 8 + g) * L.ars + kk;
                    mma_bf16_16816(d, lds32(x0), lds32(x1), lds32(x0 + 8), lds32(x1 + 8), lds32(ar), lds32(ar + 8));
                }
                float *p = sP + g * prs + cb * 8 + 2 * q;
                atomicAdd(p, d[0]);
                atomicAdd(p + 1, d[1]);
                atomicAdd(p + 8 * prs, d[2]);
                atomicAdd(p + 8 * prs + 1, d[3]);
            }
        }
        __syncthreads();
        cluster_sync();  // every CTA's partial is complete

        // ---- the KS partials of this CTA's share of (token, rank), in rank order,
        // as bf16 hi + lo into the sums tiles of every CTA ----
        {
            const int32_t E = len * prs;
            const int32_t e_lo = static_cast<int32_t>(static_cast<int64_t>(c) * E / KS);
            const int32_t e_hi = static_cast<int32_t>(static_cast<int64_t>(c + 1) * E / KS);
            for (int32_t e = e_lo + tid; e < e_hi; e += kCThreads) {
                const int32_t row = e / prs, col = e % prs, i = col / L.rp8, j = col % L.rp8;
                if (j >= r) continue;
                const uint32_t off = base + L.p_off + static_cast<uint32_t>(e * 4);
                float acc = 0.f;
                for (uint32_t rr = 0; rr < KS; ++rr) acc += ld_dsmem_f32(map_to_rank(off, rr));
                const uint16_t hi = bf16_bits(acc);
                const uint16_t lo = bf16_bits(acc - __uint_as_float(static_cast<uint32_t>(hi) << 16));
                const uint32_t so = base + L.s_off + static_cast<uint32_t>((row * L.srs + i * L.rp16 + j) * 2);
                const uint32_t so_lo = so + static_cast<uint32_t>(kCTok * L.srs * 2);
                for (uint32_t rr = 0; rr < KS; ++rr) {
                    st_dsmem_u16(map_to_rank(so, rr), hi);
                    st_dsmem_u16(map_to_rank(so_lo, rr), lo);
                }
            }
        }
        cluster_sync();  // the sums are in every CTA; no partial is read any more

        // ---- expand: 8-column blocks of the CTA's columns; y updated in the tile ----
        {
            const int32_t nblk = L.ncol / 8, ksteps = (r + 15) / 16;
            for (int32_t bk = warp; bk < nblk; bk += kCThreads / 32) {
                int32_t i = 0, colbase = 0, dci = 0, w = 0;
                for (;; ++i) {
                    const int32_t di = sh.off[i + 1] - sh.off[i];
                    dci = slice_share(di, static_cast<int32_t>(KS));
                    const int32_t mc0 = static_cast<int32_t>(c) * dci;
                    w = max(0, min(di, mc0 + dci) - mc0);
                    if (bk * 8 < colbase + dci || i + 1 == sh.n) break;
                    colbase += dci;
                }
                if (bk * 8 - colbase >= w) continue;  // columns past the slice
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                for (int32_t ks = 0; ks < ksteps; ++ks) {
                    const int32_t kk = i * L.rp16 + ks * 16 + 2 * q;
                    const uint16_t *h0 = sHi + g * L.srs + kk, *h1 = h0 + 8 * L.srs;
                    const uint16_t *l0 = sLo + g * L.srs + kk, *l1 = l0 + 8 * L.srs;
                    const uint16_t *br = sB + (bk * 8 + g) * L.brs + ks * 16 + 2 * q;
                    const uint32_t b0 = lds32(br), b1 = lds32(br + 8);
                    mma_bf16_16816(d, lds32(h0), lds32(h1), lds32(h0 + 8), lds32(h1 + 8), b0, b1);
                    mma_bf16_16816(d, lds32(l0), lds32(l1), lds32(l0 + 8), lds32(l1 + 8), b0, b1);
                }
                const int32_t col = bk * 8 + 2 * q;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int32_t row = g + 8 * h;
                    if (row < len) {
                        uint32_t *yp = reinterpret_cast<uint32_t *>(sY + row * L.yrs + col);
                        const uint32_t yv = *yp;
                        *yp = pack_bf16x2(bf16lo_to_f32(yv) + scale * d[2 * h], bf16hi_to_f32(yv) + scale * d[2 * h + 1]);
                    }
                }
            }
        }
        __syncthreads();

        // ---- the updated rows back: 16-byte pieces ----
        {
            int32_t colbase = 0;
            for (int i = 0; i < sh.n; ++i) {
                const int32_t di = sh.off[i + 1] - sh.off[i], dci = slice_share(di, static_cast<int32_t>(KS));
                const int32_t mc0 = static_cast<int32_t>(c) * dci, w = max(0, min(di, mc0 + dci) - mc0);
                const int32_t ych = w / 8;
                for (int32_t e = tid; e < len * ych; e += kCThreads) {
                    const int32_t row = e / ych, ch = e % ych, t = s_tok[row];
                    if (t >= 0)
                        stg_u4(a.y + static_cast<int64_t>(t) * a.ldy + sh.off[i] + mc0 + ch * 8,
                               *reinterpret_cast<const uint4 *>(sY + row * L.yrs + colbase + ch * 8));
                }
                colbase += dci;
            }
        }
        __syncthreads();  // the next chunk refills the x, y and token tiles
    }
}

// Cluster size: 16 CTAs (twice the copy streams of 8, measured faster on a
// 64-token q_proj call; a CTA's tiles only shrink as the cluster grows, so a
// shape that does not fit 16 fits no smaller cluster either); 0: unsupported.
int32_t cluster_size_for(const Shape &sh) {
    return c_layout(sh, 16).bytes <= static_cast<uint32_t>(kCSmemLimit) ? 16 : 0;
}

}  // namespace

bool cluster_decode_supported(int32_t T, const Shape &sh) {
    if (T < 1 || sh.k < 8 || sh.k % 8 != 0 || sh.r_max > 256) return false;
    for (int i = 0; i <= sh.n; ++i)
        if (sh.off[i] % 8 != 0) return false;
    return cluster_size_for(sh) > 0;
}

cudaError_t launch_cluster_decode(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                  const void *table, const int32_t *sorted_ids, const int32_t *seg, int32_t T,
                                  int32_t *err, cudaStream_t stream, int32_t xdiv) {
    if (!cluster_decode_supported(T, sh) || xdiv < 1 || T % xdiv != 0) return cudaErrorNotSupported;
    const int32_t KS = cluster_size_for(sh);
    const CLayout L = c_layout(sh, KS);
    cudaError_t e = cudaFuncSetAttribute(cluster_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L.bytes));
    if (e != cudaSuccess) return e;
    if (KS > 8) {
        e = cudaFuncSetAttribute(cluster_decode_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    CArgs a{x, ldx, y, ldy, table, sorted_ids, seg, err, T, xdiv};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(KS), static_cast<unsigned>(sh.S));
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = L.bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(KS);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, cluster_decode_kernel, a, sh);
}

}  // namespace lora
