// Device-side helpers shared by the library's kernels (not by the oracle).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/lora_gemm.h"

namespace lora {

// ---------------------------------------------------------------------------
// Packed slot table (device memory, caller-owned).  Layout, 16-byte aligned:
//   [0, 16)            int32 magic, S, n_slices, r_max
//   rank_off           int32 rank[S]            (padded to 16 bytes)
//   scale_off          float scale[S]           (padded to 16 bytes)
//   a_off              uint64 A[S * n_slices]   (slot-major)
//   b_off              uint64 B[S * n_slices]
// ---------------------------------------------------------------------------
constexpr int32_t kTableMagic = 0x41526f4c;  // "LoRA"
// Set in header word 3 (r_max, which no kernel reads) of a table whose tensor
// maps follow it: the only reader of those maps checks this bit before it reads
// anything past the plain table.
constexpr int32_t kTableMapsFlag = 1 << 30;

__host__ __device__ inline size_t pad16(size_t b) { return (b + 15) & ~size_t(15); }

struct TableLayout {
    size_t rank_off, scale_off, a_off, b_off, bytes;
    __host__ __device__ TableLayout(int32_t S, int32_t n) {
        rank_off = 16;
        scale_off = rank_off + pad16(sizeof(int32_t) * size_t(S));
        a_off = scale_off + pad16(sizeof(float) * size_t(S));
        b_off = a_off + sizeof(uint64_t) * size_t(S) * size_t(n);
        bytes = b_off + sizeof(uint64_t) * size_t(S) * size_t(n);
    }
};

struct TableView {
    const int32_t *rank;
    const float *scale;
    const uint64_t *a_ptr;
    const uint64_t *b_ptr;
    int32_t S, n;
    __host__ __device__ TableView(const void *base, int32_t S_, int32_t n_) : S(S_), n(n_) {
        TableLayout L(S_, n_);
        const char *p = static_cast<const char *>(base);
        rank = reinterpret_cast<const int32_t *>(p + L.rank_off);
        scale = reinterpret_cast<const float *>(p + L.scale_off);
        a_ptr = reinterpret_cast<const uint64_t *>(p + L.a_off);
        b_ptr = reinterpret_cast<const uint64_t *>(p + L.b_off);
    }
};

// Rank padding of the tensor-core prefill path: 16, 32 or 64 columns (rows of
// 32, 64 or 128 bytes, one swizzle span).
__host__ __device__ inline int32_t tc_rank_pad(int32_t r_max) { return r_max <= 16 ? 16 : (r_max <= 32 ? 32 : 64); }

// Plan of the one-kernel TMA decode path: a 128-byte header, 64 bytes per
// slot, 32 bytes for each of up to 512 CTAs, then the T sorted token ids.
__host__ __device__ inline size_t tma_plan_size(int32_t T, int32_t S) {
    return (128 + 64 * size_t(S) + 512 * 32 + 4 * size_t(T > 0 ? T : 0) + 255) & ~size_t(255);
}

// Workspace: a control block of per-(slot, slice) counters, the fp32 xa that
// lora_shrink writes (and lora_expand reads), the fp32 accumulator of the
// fused decode kernel, which every call leaves zeroed for the next one, and
// (r_max <= 64) the prefill path's xa as bf16 hi and lo parts, [n][T][RP] each
// in sorted-token order.  Then, for r_max <= 64, the one-kernel TMA decode
// path's two fp32 sum sets (the size of xa, used in turn), its control block
// (2 S per-slot counters, the call counter and the exit counter) and room for
// the plan a call without one builds.
struct WorkspaceLayout {
    size_t ctrl_bytes, xa_off, acc_off, hi_off, lo_off, acc2_off, acc3_off, tacc0_off, tacc1_off, tctrl_off,
        tplan_off, bytes;
    __host__ __device__ WorkspaceLayout(int32_t T, int32_t n_slices, int32_t r_max, int32_t S) {
        // two int32 counters per (slot, slice) + a few global words, rounded to 256 B
        ctrl_bytes = (sizeof(int32_t) * (2 * size_t(S) * LORA_MAX_SLICES + 64) + 255) & ~size_t(255);
        const size_t tt = size_t(T > 0 ? T : 0);
        const size_t xa_bytes = sizeof(float) * size_t(n_slices) * tt * size_t(r_max);
        const bool tc = r_max <= 64;  // the tensor-core paths' extra regions
        const size_t hl_bytes = tc ? sizeof(uint16_t) * size_t(n_slices) * tt * size_t(tc_rank_pad(r_max)) : 0;
        xa_off = ctrl_bytes;
        acc_off = xa_off + ((xa_bytes + 255) & ~size_t(255));
        hi_off = acc_off + ((xa_bytes + 255) & ~size_t(255));
        lo_off = hi_off + ((hl_bytes + 255) & ~size_t(255));
        // two more fp32 accumulators, used in turn by the two-kernel decode paths
        const size_t acc_tc = r_max <= 128 ? ((xa_bytes + 255) & ~size_t(255)) : 0;
        acc2_off = lo_off + ((hl_bytes + 255) & ~size_t(255));
        acc3_off = acc2_off + acc_tc;
        const size_t xa_r = (xa_bytes + 255) & ~size_t(255);
        tacc0_off = acc3_off + acc_tc;
        tacc1_off = tacc0_off + (tc ? xa_r : 0);
        tctrl_off = tacc1_off + (tc ? xa_r : 0);
        tplan_off = tctrl_off + (tc ? ((sizeof(int32_t) * (2 * size_t(S) + 2) + 255) & ~size_t(255)) : 0);
        bytes = tplan_off + (tc ? tma_plan_size(T, S) : 0);
    }
};

// Shape passed by value to kernels.
struct Shape {
    int32_t S, r_max, k, n;
    int32_t off[LORA_MAX_SLICES + 1];
};

// ---------------------------------------------------------------------------
// Error reporting: first error wins, the word is never cleared here.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report_error(int32_t *err, int32_t code) {
    if (err != nullptr) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// Memory access
// ---------------------------------------------------------------------------
// Read-only 16-byte load through the non-coherent path, no L1 allocation: for
// weights and activations streamed once per call.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Coherent 16-byte load (data written earlier in the same kernel by other CTAs).
__device__ __forceinline__ uint4 ldg_cg(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ldg_cg_f4(const float *p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void stg_u4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ int32_t ld_acquire(const int32_t *p) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// bf16 helpers (bit-level; a bf16 is the high half of an fp32)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> packed bf16x2 (lo in the low half), round-to-nearest-even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core MMA (m16n8k16, bf16 in, fp32 accumulate).
// Fragment ownership for lane = 4*g + q:
//   A (16x16, row-major): a0 = (row g, k 2q..2q+1), a1 = (row g+8, k 2q..),
//                         a2 = (row g, k 2q+8..),   a3 = (row g+8, k 2q+8..)
//   B (16x8,  col-major): b0 = (k 2q..2q+1, col g), b1 = (k 2q+8.., col g)
//   C/D (16x8, fp32):     d0,d1 = (row g, cols 2q, 2q+1), d2,d3 = (row g+8, cols 2q, 2q+1)
// ---------------------------------------------------------------------------
// Not volatile: a pure register operation, so the compiler may interleave
// independent MMAs and loads.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// Block-wide scan
// ---------------------------------------------------------------------------
// Exclusive scan of smem[0..n) in place with all threads of the block; returns
// the total.  scratch needs blockDim/32 + 1 ints.
static __device__ __noinline__ int32_t block_exclusive_scan(int32_t *data, int32_t n, int32_t *scratch) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int32_t local = 0;
    for (int e = lo; e < hi; ++e) local += data[e];
    int32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = nt >> 5;
        int32_t v = lane < nw ? scratch[lane] : 0;
        int32_t w_incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t u = __shfl_up_sync(0xffffffffu, w_incl, o);
            if (lane >= o) w_incl += u;
        }
        if (lane < nw) scratch[lane] = w_incl - v;  // exclusive warp offsets
        if (lane == nw - 1) scratch[32] = w_incl;    // total
    }
    __syncthreads();
    int32_t run = scratch[warp] + incl - local;
    for (int e = lo; e < hi; ++e) {
        int32_t v = data[e];
        data[e] = run;
        run += v;
    }
    int32_t total = scratch[32];
    __syncthreads();
    return total;
}


// ---------------------------------------------------------------------------
// Thread-block clusters and distributed shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// Work items over slots
// ---------------------------------------------------------------------------
// Per-slot work items, computed by the whole block: s_pref[s] becomes the
// exclusive prefix of items(n_s, r_s) over slots with tokens and rank > 0.
// Guards: the table header must match the shape, the index must cover exactly
// T tokens and no rank may exceed r_max (the workspace row stride); otherwise
// the offending work is dropped and the error word set.
template <class F>
__device__ int32_t slot_item_prefix(const void *table, const Shape &sh, const int32_t *seg, int32_t T,
                                    int32_t *s_pref, int32_t *s_scr, int32_t *err, F items) {
    const int32_t *hdr = static_cast<const int32_t *>(table);
    const TableView tab(table, sh.S, sh.n);
    const bool ok = hdr[0] == kTableMagic && hdr[1] == sh.S && hdr[2] == sh.n && seg[sh.S + 1] == T;
    if (!ok && threadIdx.x == 0 && blockIdx.x == 0) report_error(err, LORA_ERR_INVALID_ARG);
    for (int s = threadIdx.x; s < sh.S; s += blockDim.x) {
        const int32_t n = ok ? seg[s + 1] - seg[s] : 0;
        const int32_t r = ok ? tab.rank[s] : 0;
        const bool rank_ok = r <= sh.r_max;
        if (!rank_ok && blockIdx.x == 0) report_error(err, LORA_ERR_RANK);
        s_pref[s] = (ok && rank_ok && n > 0 && r > 0) ? items(n, r) : 0;
    }
    __syncthreads();
    return block_exclusive_scan(s_pref, sh.S, s_scr);
}

// Slot owning item u: the last slot whose exclusive prefix is <= u.
__device__ __forceinline__ int32_t find_slot(const int32_t *s_pref, int32_t S, int32_t u) {
    int32_t lo = 0, hi = S;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (s_pref[mid] <= u) lo = mid + 1;
        else hi = mid;
    }
    return lo - 1;
}

// fp32 pair -> bf16 hi part and bf16 remainder (v = hi + lo to ~2^-17 relative).
__device__ __forceinline__ void split_bf16x2(float v0, float v1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16x2(v0, v1);
    lo = pack_bf16x2(v0 - bf16lo_to_f32(hi), v1 - bf16hi_to_f32(hi));
}

}  // namespace lora
