// Per-step token index: a stable counting sort of tokens by adapter slot.
//
// TensorRT-LLM LoRA serving page, section "一次 decode 批次的路由" (steps 2 and 4:
// sorted ids, bincount over slots, cumsum with one extra entry holding the
// total) and vLLM book ch. 16, section 16.4.3 (LoRAKernelMeta: tokens sorted by
// slot, tokens per slot, segment starts, active slots).  No-adapter tokens
// (slot -1) and out-of-range ids are keyed S, i.e. placed last, like
// TensorRT-LLM's sentinel slot after the real ones.
//
// Speculative decoding (TensorRT-LLM LoRA serving page, "一次 decode 批次的路由":
// tokens_per_seq > 1 expands the sequence order to the token order as
// sorted * tokens_per_seq + arange(tokens_per_seq)): the keys are one per
// sequence, sequence b owning tokens b tps .. b tps + tps - 1; the counts are
// multiplied by tps and each sequence writes its tps token ids in a row.  With
// tps = 1 this is the token-level sort.
//
// Routed-expert (MoE) LoRA (llama.cpp LoRA adapter page, "MoE 专属的
// build_lora_mm_id": A and B are routed by the same expert ids as the base
// weights; TensorRT-LLM LoRA serving page, "MoE LoRA": one (A, B) pair per
// expert): the keys are (token, choice) pairs p = t K + j, pair p of a token
// with adapter s routed to expert e = expert_ids[p] has the virtual slot
// s E + e of a table of S = n_adapters E slots, and is keyed S when the token
// has no adapter.
//
// Activated LoRA (llama.cpp LoRA adapter page, "aLoRA:让适配器在 prompt 中间生效":
// a request runs without its adapter up to the invocation point and with it
// from there on): with seq_ids given, token t of sequence q = seq_ids[t] at
// position positions[t] is keyed seq_slot[q] when positions[t] >=
// invocation_start[q] and S (no adapter) before it.
//
// One thread block does the whole sort: histogram in shared memory, an
// exclusive scan into the segment offsets, then a pass over the tokens in
// blockDim-sized chunks in token order.  Inside a chunk, a token's place among
// equal keys is its rank within its warp (__match_any_sync + popc) plus the
// counts of the same key in lower warps; the running per-key cursor carries
// the order across chunks, so ties stay in ascending token index.
#include "common.cuh"

namespace lora {

namespace {

// Per-token activation of aLoRA: sequence ids and positions of the tokens, the
// sequences' slots and invocation starts.
struct Activation {
    const int32_t *seq_ids, *positions, *seq_slot, *invocation_start;
    int32_t n_seq;
};

// Key of item t: its slot, or S for no adapter or an id out of range (bad).
// With expert_ids, item t is the pair (t / K, t % K) and its key the virtual
// slot slot_ids[t / K] * E + expert_ids[t].  With act.seq_ids, the slot of
// token t is its sequence's from the invocation start on.
__device__ __forceinline__ int32_t index_key(const int32_t *__restrict__ slot_ids,
                                             const int32_t *__restrict__ expert_ids, const Activation &act,
                                             int32_t t, int32_t K, int32_t E, int32_t S, bool &bad) {
    if (act.seq_ids != nullptr) {
        const int32_t q = act.seq_ids[t];
        if (q < 0 || q >= act.n_seq) {
            bad = true;
            return S;
        }
        const int32_t s = act.positions[t] >= act.invocation_start[q] ? act.seq_slot[q] : -1;
        bad |= (s < -1 || s >= S);
        return (s >= 0 && s < S) ? s : S;
    }
    if (expert_ids == nullptr) {
        const int32_t s = slot_ids[t];
        bad |= (s < -1 || s >= S);
        return (s >= 0 && s < S) ? s : S;
    }
    const int32_t s = slot_ids[t / K], e = expert_ids[t], SA = S / E;
    const bool ok = s >= 0 && s < SA && e >= 0 && e < E;
    bad |= (s < -1 || s >= SA || (s >= 0 && !ok));
    return ok ? s * E + e : S;
}

__global__ void build_index_kernel(const int32_t *__restrict__ slot_ids, const int32_t *__restrict__ expert_ids,
                                   Activation act, int32_t T, int32_t tps, int32_t K, int32_t E, int32_t S,
                                   const void *table,
                                   int32_t *__restrict__ sorted_ids, int32_t *__restrict__ seg_offsets,
                                   int32_t *__restrict__ active, int32_t *err) {
    extern __shared__ int32_t smem[];
    const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = nt >> 5;
    const int bins = S + 1;
    int32_t *cursor = smem;              // [bins]   histogram, then running cursor
    int32_t *flag = cursor + bins;       // [S]      active flags, then positions
    int32_t *wcnt = flag + S;            // [bins * nw] per-chunk per-warp counts
    int32_t *scratch = wcnt + bins * nw; // [33]

    const TableView tab(table, S, 1);
    const int32_t *hdr = static_cast<const int32_t *>(table);
    const bool table_ok = hdr[0] == kTableMagic && hdr[1] == S;  // else ranks are not read at all
    if (tid == 0 && !table_ok) report_error(err, LORA_ERR_INVALID_ARG);
    for (int b = tid; b < bins; b += nt) cursor[b] = 0;
    for (int e = tid; e < bins * nw; e += nt) wcnt[e] = 0;
    __syncthreads();

    // 1. histogram
    bool bad = false;
    for (int t = tid; t < T; t += nt) atomicAdd(&cursor[index_key(slot_ids, expert_ids, act, t, K, E, S, bad)], tps);
    if (bad) report_error(err, LORA_ERR_SLOT_RANGE);
    __syncthreads();

    // 2. active slots: tokens present and rank > 0, ascending
    for (int s = tid; s < S; s += nt) flag[s] = (table_ok && cursor[s] > 0 && tab.rank[s] > 0) ? 1 : 0;
    __syncthreads();
    {
        // the scan turns flags into positions; activity is re-derived from the counts
        int32_t n_active = block_exclusive_scan(flag, S, scratch);
        for (int s = tid; s < S; s += nt) {
            const bool is_active = table_ok && cursor[s] > 0 && tab.rank[s] > 0;
            if (is_active) active[1 + flag[s]] = s;
        }
        if (tid == 0) active[0] = n_active;
    }

    // 3. segment offsets
    block_exclusive_scan(cursor, bins, scratch);
    for (int b = tid; b < bins; b += nt) seg_offsets[b] = cursor[b];
    if (tid == 0) seg_offsets[S + 1] = T * tps;
    __syncthreads();

    // 4. stable scatter, chunk by chunk in token order
    for (int base = 0; base < T; base += nt) {
        const int t = base + tid;
        const bool valid = t < T;
        int32_t key = -1 - lane;  // unique per lane for invalid tokens: never matches
        bool unused = false;
        if (valid) key = index_key(slot_ids, expert_ids, act, t, K, E, S, unused);
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const unsigned lower = peers & ((1u << lane) - 1u);
        const int in_warp = __popc(lower);
        const bool leader = lower == 0;
        if (valid && leader) wcnt[key * nw + warp] = __popc(peers);
        __syncthreads();
        if (valid) {
            int32_t before = 0;
            for (int w = 0; w < warp; ++w) before += wcnt[key * nw + w];
            int32_t *dst = sorted_ids + cursor[key] + (before + in_warp) * tps;
            for (int32_t j = 0; j < tps; ++j) dst[j] = t * tps + j;
        }
        __syncthreads();
        if (valid && leader) {
            atomicAdd(&cursor[key], __popc(peers) * tps);
            wcnt[key * nw + warp] = 0;
        }
        __syncthreads();
    }
}

}  // namespace

size_t index_smem_bytes(int32_t S, int threads) {
    const int nw = threads / 32;
    return sizeof(int32_t) * (size_t(S + 1) + size_t(S) + size_t(S + 1) * nw + 33);
}

// T keys (tokens, sequences of tps tokens each, or with expert_ids (K, E)
// token-expert pairs).
cudaError_t launch_build_index(const int32_t *slot_ids, const int32_t *expert_ids, int32_t T, int32_t tps, int32_t K,
                               int32_t E, int32_t S, const void *table, int32_t *sorted_ids, int32_t *seg_offsets,
                               int32_t *active, int32_t *err, cudaStream_t stream, const int32_t *seq_ids,
                               const int32_t *positions, const int32_t *seq_slot, const int32_t *invocation_start,
                               int32_t n_seq) {
    const Activation act{seq_ids, positions, seq_slot, invocation_start, n_seq};
    int threads = 1024;
    if (T < 1024) threads = ((T + 31) / 32) * 32;
    if (threads < 128) threads = 128;
    size_t smem = index_smem_bytes(S, threads);
    while (smem > 200 * 1024 && threads > 128) {
        threads /= 2;
        smem = index_smem_bytes(S, threads);
    }
    // per call: the attribute belongs to the current device's context
    cudaError_t ea = cudaFuncSetAttribute(build_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          200 * 1024);
    if (ea != cudaSuccess) return ea;
    build_index_kernel<<<1, threads, smem, stream>>>(slot_ids, expert_ids, act, T, tps, K, E, S, table, sorted_ids,
                                                     seg_offsets, active, err);
    return cudaGetLastError();
}

}  // namespace lora
