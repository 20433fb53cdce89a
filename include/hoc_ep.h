/*
 * hoc_ep.h -- expert-parallel pack and combine around the dispatch / combine
 * all-to-all (HOCCL section 2.1 and Table 1: EP token dispatch and combine are
 * all-to-all traffic).  Device pointers, stream-ordered, no host
 * synchronisation, so the counts can feed hoc_alltoall_device_counts directly.
 */
#ifndef HOC_EP_H
#define HOC_EP_H

#include <stddef.h>
#include <stdint.h>

#include "hoc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Dispatch-side pack of one source rank.  expert_ids: [tokens*topk] int32
 * (pair j of token t at t*topk + j); x: [tokens, hidden] bf16 token rows.
 * Experts e = 0..experts-1 live on rank e / (experts / nranks).  Writes
 *   send:       the rows of the valid pairs ordered by (destination rank,
 *               expert, token, slot), [tokens*topk, hidden] bf16 capacity;
 *   perm[i]:    t*topk + j of the pair in row i (-1 past the valid pairs);
 *   pos_of[p]:  the row of pair p (-1 for a dropped pair);
 *   dst_counts: [nranks] uint64 elements (rows * hidden) per destination.
 * workspace: device int32 scratch of workspace_ints entries, at least what
 * hoc_ep_pack_workspace() returns (else HOC_ERR_INVALID_ARG, nothing queued).
 * Pairs with an expert id outside [0, experts) are dropped.  experts must be a
 * multiple of nranks.  With tokens == 0 only dst_counts is written (all 0).  The sort is a stable counting sort over tiles of 2048
 * pairs (tile histograms, one scan, stable placement by warp match); with more
 * than 1024 experts one CTA per expert scans every pair instead. */
hocResult_t hoc_ep_pack(const int32_t* expert_ids, const void* x, int tokens, int topk, int hidden, int experts,
                        int nranks, void* send, int32_t* perm, int32_t* pos_of, uint64_t* dst_counts,
                        int32_t* workspace, size_t workspace_ints, void* stream);

/* int32 entries of the workspace hoc_ep_pack needs for this shape. */
hocResult_t hoc_ep_pack_workspace(int tokens, int topk, int experts, size_t* ints);

/* Combine (unpack) of one source rank after the inverse exchange.  rows:
 * [tokens*topk, hidden] bf16 in packed order; pos_of from hoc_ep_pack;
 * weights: [tokens*topk] fp32 gate weights.  y[t] = bf16 of the binary32 fold,
 * in slot order, of fp32(weights[t*topk+j] * row[pos_of[t*topk+j]]) over the
 * token's valid pairs (products and sums rounded to nearest even, no fused
 * multiply-add; +0 when no pair is valid). */
hocResult_t hoc_ep_combine(const void* rows, const int32_t* pos_of, const float* weights, int tokens, int topk,
                           int hidden, void* y, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* HOC_EP_H */
