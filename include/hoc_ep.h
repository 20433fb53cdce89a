/*
 * hoc_ep.h -- expert-parallel pack and combine around the dispatch / combine
 * all-to-all (HOCCL section 2.1 and Table 1: EP token dispatch and combine are
 * all-to-all traffic).  Device pointers, stream-ordered, no host
 * synchronisation, so the counts can feed hoc_alltoall_device_counts directly.
 * Every call here may be captured into a CUDA graph and replayed on new data
 * in the same buffers (the sort, the counts and the row positions are
 * recomputed on the device at each replay); make one call of each kind before
 * the capture, so that its kernels are loaded and their attributes set.
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
 * multiply-add; +0 when no pair is valid).  Runs on register-fed vector loads
 * and has no status word, so it never waits on anything; hoc_ep_combine_all
 * (nranks = 1 for one rank) gives the same bits on the faster TMA-fed kernel,
 * with a status word for its bounded waits and row checks. */
hocResult_t hoc_ep_combine(const void* rows, const int32_t* pos_of, const float* weights, int tokens, int topk,
                           int hidden, void* y, void* stream);

/* ---------------------------------------------------------------------------
 * Dispatch and combine fused with the all-to-all.  All k simulated ranks live
 * in one GPU's memory, so no send buffer and no exchange is needed: the row
 * scatter writes every token row straight to the place in the destination
 * rank's receive buffer that the dispatch all-to-all (default displacements:
 * prefix sums in rank order) would have copied it to, and the combine reads a
 * token's top-k rows straight from the expert ranks' buffers, where the
 * inverse exchange would have fetched them.  Both run on SMs; the copy-engine
 * exchange (hoc_ep_pack + hoc_alltoall_device_counts + hoc_ep_combine) stays
 * the zero-SM way.  Results are bit for bit those of pack -> all-to-all ->
 * inverse all-to-all -> combine.  Every rank has `tokens` tokens; all pointer
 * arrays are host arrays of nranks (1..HOC_MAX_RANKS) device pointers, read
 * during the call.
 * ------------------------------------------------------------------------- */

/* Dispatch of every source rank in one pass.  expert_ids[s]: [tokens*topk]
 * int32; x[s]: [tokens, hidden] bf16; recv[d]: receive buffer of rank d, room
 * for recv_capacity[d] elements (host array).  Writes
 *   recv[d]:   the rows bound for rank d, source by source, each source's rows
 *              in (expert, token, slot) order -- the layout of hoc_ep_pack's
 *              send buffers after the all-to-all;
 *   pos_of[s]: [tokens*topk] int32, the packed row of each pair of source s
 *              (-1 for a dropped pair), as hoc_ep_pack;
 *   counts:    device [nranks*nranks] uint64 element counts, row = source;
 *   *status:   device int32, cleared first; bit 0 set if a row did not fit its
 *              receive buffer (that row is not written).
 * workspace: device int32 scratch of at least nranks * hoc_ep_pack_workspace()
 * entries (else HOC_ERR_INVALID_ARG, nothing queued).  Pairs with an expert id
 * outside [0, experts) are dropped; experts is a multiple of nranks.  Stream-
 * ordered; the host does not wait.  Each token row is read once and stored
 * to each of its pairs' rows by per-thread 16-byte vector copies (rows and
 * buffers aligned to 16 bytes; byte copies otherwise).  HOC_EP_DISPATCH=bulk
 * selects TMA bulk copies through shared memory instead (one bulk load per
 * row, one bulk store per pair; topk <= 16), equally fast on GB300; bit 2 of
 * *status is set if one of that kernel's bounded waits gave up. */
hocResult_t hoc_ep_dispatch_fused(int nranks, const int32_t* const* expert_ids, const void* const* x, int tokens,
                                  int topk, int hidden, int experts, void* const* recv, const size_t* recv_capacity,
                                  int32_t* const* pos_of, uint64_t* counts, int32_t* workspace,
                                  size_t workspace_ints, int32_t* status, void* stream);

/* Combine of every source rank in one pass, reading rows[d] -- rank d's rows
 * after its experts, in the receive layout the dispatch wrote, room for
 * rows_capacity[d] elements -- at the places the dispatch's counts give.
 * expert_ids, pos_of and counts are those of the dispatch; weights[s]:
 * [tokens*topk] fp32 gate weights; y[s]: [tokens, hidden] bf16 output.  The
 * fold is hoc_ep_combine's: y[s][t] = bf16 of the binary32 sum, in slot order,
 * of fp32(weight * row) over the token's valid pairs (+0 when none).  Bit 1 of
 * *status (not cleared here) is set if a row lies outside its buffer (it then
 * adds nothing).  With hidden % 8 == 0, 16-byte-aligned rows and outputs and
 * topk <= 8, each warp's rows arrive by TMA bulk copies into shared memory
 * (two stages per warp of topk row slices, 4 KiB at topk 1, 2 KiB at topk 2-3,
 * 1 KiB from topk 4 on; bit 2 of *status if a bounded wait gave up);
 * HOC_EP_COMBINE=lsu selects per-thread vector loads instead. */
hocResult_t hoc_ep_combine_fused(int nranks, const void* const* rows, const size_t* rows_capacity,
                                 const int32_t* const* expert_ids, const int32_t* const* pos_of,
                                 const uint64_t* counts, const float* const* weights, int tokens, int topk,
                                 int hidden, int experts, void* const* y, int32_t* status, void* stream);

/* ---------------------------------------------------------------------------
 * The same pack and combine for every rank in one pass, around the copy-engine
 * exchange (hoc_alltoall_device_counts): the zero-SM way of moving the rows,
 * with the SM work of all k ranks in one set of launches instead of k.
 * ------------------------------------------------------------------------- */

/* hoc_ep_pack for every source rank at once: send[s] receives source s's rows
 * in (destination rank, expert, token, slot) order -- what hoc_ep_pack writes
 * -- with room for send_capacity[s] elements (host array; a row past it is not
 * written and sets bit 0 of *status, which is cleared first); pos_of[s] and
 * row s of counts (device [nranks*nranks] uint64 elements) as hoc_ep_pack.  No
 * perm is written.  workspace: nranks * hoc_ep_pack_workspace() int32 entries.
 * The row scatter engine follows HOC_EP_DISPATCH as for hoc_ep_dispatch_fused. */
hocResult_t hoc_ep_pack_all(int nranks, const int32_t* const* expert_ids, const void* const* x, int tokens, int topk,
                            int hidden, int experts, void* const* send, const size_t* send_capacity,
                            int32_t* const* pos_of, uint64_t* counts, int32_t* workspace, size_t workspace_ints,
                            int32_t* status, void* stream);

/* hoc_ep_combine for every source rank at once: rows[s] holds source s's rows
 * back from the experts in packed order (room for rows_capacity[s] elements;
 * a row past it adds nothing and sets bit 1 of *status, not cleared here);
 * pos_of[s], weights[s] and y[s] as hoc_ep_combine.  The engine follows
 * HOC_EP_COMBINE as for hoc_ep_combine_fused. */
hocResult_t hoc_ep_combine_all(int nranks, const void* const* rows, const size_t* rows_capacity,
                               const int32_t* const* pos_of, const float* const* weights, int tokens, int topk,
                               int hidden, void* const* y, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* HOC_EP_H */
