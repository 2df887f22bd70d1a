// Host-side planning for absorbed MLA decode: argument checks, the split count
// S, the kernel variant and the workspace layout. No CUDA calls happen here,
// so everything in this file also runs on a machine without a GPU.
#include <algorithm>
#include <cstring>
#include <functional>
#include <queue>
#include <vector>

#include "mla_internal.h"

namespace mla {

namespace {

uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Makespan of items (costs in launch order) greedily placed on `machines`
// identical workers, which is how the block scheduler hands out CTAs.
double list_schedule(const std::vector<double>& costs, int machines) {
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < machines; ++i) free_at.push(0.0);
    double makespan = 0.0;
    for (double c : costs) {
        double t = free_at.top();
        free_at.pop();
        t += c;
        makespan = std::max(makespan, t);
        free_at.push(t);
    }
    return makespan;
}

int heads_per_simt_cta() { return 16; }

// Fixed cost of one work item (or one segment of the balanced schedule) of the
// tensor-core kernel, in pages: q staging, pipeline fill and the epilogue.
constexpr double kTcItemPages = 4.0;

// Workspace layout for a plan: status header, then the partial rows and
// their fp32 LSEs. Split schedule: [B, N, S, Lkv] (bf16, or fp32 with
// MLA_PLAN_FP32_PARTIALS) and [B, N, S] (S > 1 only); balanced schedule:
// [2 * pairs, N, Lkv] fp32 and [2 * pairs, N].
void workspace_layout(int batch, int num_heads, int S, int pairs, uint32_t flags,
                      uint64_t* part_off, uint64_t* lse_off, uint64_t* bytes) {
    uint64_t rows = 0;
    uint64_t elem = sizeof(float);
    if (pairs > 0) {
        rows = uint64_t(2) * pairs * num_heads;
    } else if (S > 1) {
        rows = uint64_t(batch) * num_heads * S;
        if (!(flags & MLA_PLAN_FP32_PARTIALS)) elem = 2;
    }
    uint64_t off = kStatusBytes;
    *part_off = 0;
    *lse_off = 0;
    if (rows > 0) {
        *part_off = off;
        off = align_up(off + rows * kLkv * elem, 256);
        *lse_off = off;
        off = align_up(off + rows * sizeof(float), 256);
    }
    *bytes = off;
}

// CTA pairs of the tensor-core kernel's split schedule: one per SM pair, at
// most one per (request, split) item; each walks a contiguous run of items.
int64_t tc_split_pairs(int batch, int S, int num_sms) {
    const int64_t items = int64_t(batch) * S;
    return std::min<int64_t>(items, std::max(1, num_sms / 2));
}

// Estimated run time, in units of "one page through one worker", of a split
// count S. Each (request, split) is one work item; partial results cost
// their write + read through HBM, spread over all workers.
double estimate(int kernel, int S, int batch, int num_heads, const std::vector<int>& pages,
                int num_sms) {
    int workers;
    int items_per_split;
    if (kernel == MLA_KERNEL_TC) {
        workers = std::max(1, num_sms / 2);          // one CTA pair per item
        items_per_split = 1;
    } else {
        workers = std::max(1, num_sms * 2);          // two SIMT CTAs per SM
        items_per_split = (num_heads + heads_per_simt_cta() - 1) / heads_per_simt_cta();
    }
    const double item = kernel == MLA_KERNEL_TC ? kTcItemPages : 0.15;
    std::vector<double> costs;
    costs.reserve(size_t(batch) * S * items_per_split);
    for (int b = 0; b < batch; ++b) {
        int per_split = (pages[b] + S - 1) / S;
        for (int s = 0; s < S; ++s) {
            int here = std::max(0, std::min(per_split, pages[b] - s * per_split));
            for (int i = 0; i < items_per_split; ++i) costs.push_back(item + here);
        }
    }
    double t = list_schedule(costs, workers);
    if (S > 1) {
        const double page_bytes = double(kPageSize) * kD * 2.0;
        double partial = double(batch) * num_heads * S * (kLkv * 2.0 + 4.0) * 2.0;
        double per_round = page_bytes * (kernel == MLA_KERNEL_TC ? workers : workers / 2.0);
        t += partial / per_round + 4.0;  // + the merge launch
    }
    return t;
}

// Estimated run time, same units, of the page-balanced schedule over `pairs`
// CTA pairs: an equal share of the pages, one item cost per request a pair
// touches, and the partial rows of the requests that cross range boundaries
// (at most two per pair) written and read once.
double estimate_balanced(int pairs, int batch, int num_heads, const std::vector<int>& pages) {
    double total = 0.0;
    for (int pg : pages) total += pg;
    const double segments = 1.0 + double(batch) / pairs;
    double t = total / pairs + kTcItemPages * segments;
    const double page_bytes = double(kPageSize) * kD * 2.0;
    const double partial = 2.0 * pairs * num_heads * (kLkv * 4.0 + 4.0) * 2.0;
    t += partial / (page_bytes * pairs) + 4.0;   // + the merge launch
    return t;
}

}  // namespace

int validate_plan(const mla_decode_plan_t* p) {
    if (!p) return MLA_ERR_INVALID_ARG;
    if (p->kv_lora_rank != kLkv || p->rope_dim != kRope || p->page_size != kPageSize)
        return MLA_ERR_UNSUPPORTED;
    if (p->batch < 0 || p->num_heads < 1 || p->num_heads > kMaxHeads ||
        p->max_blocks_per_seq < 1 || p->num_kv_splits < 1 ||
        p->num_kv_splits > kMaxMergeSplits)
        return MLA_ERR_INVALID_ARG;
    if (p->kernel != MLA_KERNEL_SIMT && p->kernel != MLA_KERNEL_TC) return MLA_ERR_INVALID_ARG;
    if (p->kernel == MLA_KERNEL_TC && !tc_kernel_built()) return MLA_ERR_UNSUPPORTED;
    if (p->sched_pairs < 0 || p->sched_pairs > kMaxBalancedPairs) return MLA_ERR_INVALID_ARG;
    if (p->sched_pairs > 0 && (p->kernel != MLA_KERNEL_TC || p->num_kv_splits != 1 ||
                               p->batch > kMaxBalancedBatch))
        return MLA_ERR_INVALID_ARG;
    // The launch shape and the workspace layout follow from the sizes; a plan
    // that disagrees was not made by mla_decode_plan (or was edited).
    int64_t grid;
    if (p->kernel == MLA_KERNEL_TC)
        grid = p->sched_pairs > 0 ? 2 * int64_t(p->sched_pairs)
                                  : 2 * tc_split_pairs(p->batch, p->num_kv_splits, p->num_sms);
    else
        grid = int64_t((p->num_heads + heads_per_simt_cta() - 1) / heads_per_simt_cta()) *
               p->batch * p->num_kv_splits;
    if (grid != p->grid_ctas) return MLA_ERR_INVALID_ARG;
    uint64_t part_off, lse_off, bytes;
    workspace_layout(p->batch, p->num_heads, p->num_kv_splits, p->sched_pairs, p->flags, &part_off,
                     &lse_off, &bytes);
    if (p->partial_offset != part_off || p->lse_partial_offset != lse_off ||
        p->workspace_bytes != bytes)
        return MLA_ERR_INVALID_ARG;
    return MLA_OK;
}

}  // namespace mla

using namespace mla;

extern "C" int mla_decode_plan(int batch, int num_heads, int kv_lora_rank, int rope_dim,
                               int page_size, int max_blocks_per_seq, int max_seq_len,
                               const int32_t* seq_lens_host, int num_kv_splits, int num_sms,
                               uint32_t flags, mla_decode_plan_t* plan) {
    if (!plan) return MLA_ERR_INVALID_ARG;
    if (batch < 0 || num_heads < 1 || max_blocks_per_seq < 1 || max_seq_len < 0 ||
        num_kv_splits < 0 || num_sms < 1)
        return MLA_ERR_INVALID_ARG;
    if (kv_lora_rank != kLkv || rope_dim != kRope || page_size != kPageSize ||
        num_heads > kMaxHeads)
        return MLA_ERR_UNSUPPORTED;
    if (int64_t(max_seq_len) > int64_t(max_blocks_per_seq) * page_size)
        return MLA_ERR_INVALID_ARG;
    if (num_kv_splits > kMaxMergeSplits) return MLA_ERR_UNSUPPORTED;

    std::vector<int> pages(size_t(batch), (max_seq_len + page_size - 1) / page_size);
    int max_pages = (max_seq_len + page_size - 1) / page_size;
    if (seq_lens_host) {
        max_pages = 0;
        for (int b = 0; b < batch; ++b) {
            int L = seq_lens_host[b];
            if (L < 0 || L > max_seq_len) return MLA_ERR_INVALID_ARG;
            pages[size_t(b)] = (L + page_size - 1) / page_size;
            max_pages = std::max(max_pages, pages[size_t(b)]);
        }
    }

    // The tensor-core kernel pads the heads to an M=128 tile. Even at 16
    // heads it is far ahead of the CUDA-core kernel (a page costs it ~1.3 us
    // on a CTA pair; the CUDA-core kernel, one CTA per 16 heads and split,
    // ~2.7 us), so that one runs only when asked for or when the tensor-core
    // kernel is not built.
    int kernel = MLA_KERNEL_TC;
    if ((flags & MLA_PLAN_FORCE_SIMT) || !tc_kernel_built()) kernel = MLA_KERNEL_SIMT;

    int S = num_kv_splits;
    int pairs = 0;
    if (S == 0) {
        S = 1;
        double best = 0.0;
        if (batch > 0 && max_pages > 1) {
            best = estimate(kernel, 1, batch, num_heads, pages, num_sms);
            int cap = std::min(max_pages, 64);
            for (int s = 2; s <= cap; ++s) {
                double t = estimate(kernel, s, batch, num_heads, pages, num_sms);
                if (t < best * 0.995) {
                    best = t;
                    S = s;
                }
            }
        }
        // The page-balanced schedule: every co-resident CTA pair gets an
        // equal share of the batch's pages (tensor-core kernel only).
        int64_t total_pages = 0;
        for (int pg : pages) total_pages += pg;
        const int c = int(std::min<int64_t>({int64_t(num_sms / 2), int64_t(kMaxBalancedPairs),
                                             total_pages}));
        if (kernel == MLA_KERNEL_TC && !(flags & MLA_PLAN_SPLIT_ONLY) && batch > 0 &&
            batch <= kMaxBalancedBatch && c >= 1 &&
            int64_t(batch) * max_blocks_per_seq < (int64_t(1) << 31) &&
            ((flags & MLA_PLAN_FORCE_BALANCED) ||
             (best > 0.0 && estimate_balanced(c, batch, num_heads, pages) < best * 0.98))) {
            pairs = c;
            S = 1;
        }
    }

    std::memset(plan, 0, sizeof(*plan));
    plan->batch = batch;
    plan->num_heads = num_heads;
    plan->kv_lora_rank = kv_lora_rank;
    plan->rope_dim = rope_dim;
    plan->page_size = page_size;
    plan->max_blocks_per_seq = max_blocks_per_seq;
    plan->max_seq_len = max_seq_len;
    plan->num_kv_splits = S;
    plan->sched_pairs = pairs;
    plan->kernel = kernel;
    plan->num_sms = num_sms;
    plan->flags = flags;
    if (kernel == MLA_KERNEL_TC)
        plan->grid_ctas = pairs > 0 ? 2 * pairs : int(2 * tc_split_pairs(batch, S, num_sms));
    else
        plan->grid_ctas = ((num_heads + heads_per_simt_cta() - 1) / heads_per_simt_cta()) * batch * S;

    workspace_layout(batch, num_heads, S, pairs, flags, &plan->partial_offset,
                     &plan->lse_partial_offset, &plan->workspace_bytes);
    return MLA_OK;
}

extern "C" int mla_dcp_local_seq_lens(const int32_t* seq_lens_host, int batch, int world,
                                      int rank, int interleave, int32_t* local_lens_host) {
    if (!seq_lens_host || !local_lens_host || batch < 0 || world < 1 || rank < 0 ||
        rank >= world || interleave < 1)
        return MLA_ERR_INVALID_ARG;
    for (int b = 0; b < batch; ++b)
        if (seq_lens_host[b] < 0) return MLA_ERR_INVALID_ARG;
    const int64_t span = int64_t(world) * interleave;   // one virtual block
    for (int b = 0; b < batch; ++b) {
        const int64_t L = seq_lens_host[b];
        // Whole virtual blocks give every rank `interleave` tokens; the last,
        // partial one is dealt run by run from rank 0.
        const int64_t tail = L % span - int64_t(rank) * interleave;
        const int64_t extra = tail <= 0 ? 0 : (tail < interleave ? tail : interleave);
        local_lens_host[b] = int32_t((L / span) * interleave + extra);
    }
    return MLA_OK;
}

extern "C" int mla_multi_token_row_lens(const int32_t* seq_lens_host, int batch, int q_len,
                                        int causal, int32_t* row_lens_host) {
    if (!seq_lens_host || !row_lens_host || batch < 0 || q_len < 1) return MLA_ERR_INVALID_ARG;
    for (int b = 0; b < batch; ++b)
        if (seq_lens_host[b] < 0) return MLA_ERR_INVALID_ARG;
    for (int b = 0; b < batch; ++b) {
        for (int i = 0; i < q_len; ++i) {
            // Query token i sits at position L - q_len + i and, causally,
            // sees the tokens up to and including its own position.
            const int64_t L = seq_lens_host[b];
            const int64_t seen = causal ? L - (q_len - 1 - i) : L;
            row_lens_host[int64_t(b) * q_len + i] = int32_t(seen > 0 ? seen : 0);
        }
    }
    return MLA_OK;
}

extern "C" const char* mla_status_string(int status) {
    switch (status) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported shape or kernel";
        case MLA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case MLA_ERR_CUDA: return "CUDA runtime error";
        case MLA_ERR_BAD_BLOCK_ID: return "block_table entry outside [0, num_blocks)";
        case MLA_ERR_BAD_SEQ_LEN: return "seq_len negative or beyond the block table";
        case MLA_ERR_TIMEOUT: return "bounded device wait expired";
        case MLA_ERR_SCRATCH_LIMIT:
            return "plan needs more scratch than the 32 MiB of mla_decode_noalloc";
        case MLA_ERR_RANGE: return "q entry beyond the f16 range of the fp8-cache decode";
        default: return "unknown status";
    }
}

extern "C" int mla_abi_version(void) { return MLA_DECODE_ABI_VERSION; }
