/*
 * hoc_sched.h -- two-domain stage scheduler (host only, no GPU).
 *
 * HOCCL section 3.4 ("Collective Scheduler", Fig. 6, Eqs. 2-11, Algorithm 1):
 * a collective's origin traffic matrix C (C[u*G+v] = bytes from GPU u to GPU
 * v) is expanded into the HOCCL traffic matrix T, which adds the NVLink
 * forwarding copies that carry every inter-node flow through the RDMA staging
 * buffers on each GPU's symmetric peer (Eqs. 2-5), and T is decomposed into
 * stages: each stage moves the largest removable portion of one contention-free
 * RDMA matching (at most one outgoing and one incoming inter-node flow per GPU,
 * Eq. 8) together with its forwarding copies, and fills the NVLink slack with
 * native intra-node matchings; the stages sum to T (Eq. 7).  Stage durations
 * follow Eqs. 9-10 and their sum (Eq. 11) is returned.
 *
 * Where the algorithm leaves a choice open, this implementation takes: greedy
 * matchings (largest entry first, ties by row then column); native matchings
 * peeled per NVLink domain in domain order and added to a stage's slack in
 * that order, each by the largest amount that keeps every cell of the matching
 * within tau * bw_nvlink bytes; native traffic left when the inter-node
 * traffic is exhausted runs the domains in parallel: each further stage takes
 * the next remaining matching of every domain.
 *
 * This models the multi-node schedule the paper runs on RDMA clusters; on one
 * GPU nothing executes it.  The single-domain special case (shift stages of an
 * all-to-all) is what hoc_alltoall executes.
 */
#ifndef HOC_SCHED_H
#define HOC_SCHED_H

#include <stddef.h>
#include <stdint.h>

#include "hoc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* G GPUs (1..64).  node_of[u]: NVLink domain of u.  sym[u]: u's symmetric peer,
 * a different GPU of the same node with sym[sym[u]] == u.  C: G*G bytes, row =
 * source; the diagonal must be 0.  bw_nvlink, bw_rdma: domain bandwidths in
 * bytes per time unit (positive integers).
 * Outputs (each may be NULL): T (G*G), stages (max_stages * G*G, row-major
 * stage after stage), taus (max_stages), n_stages (always written when
 * non-NULL), total (sum of the stage durations).  Returns HOC_ERR_INVALID_ARG
 * for a bad topology or matrix, HOC_ERR_OOM if more than max_stages stages
 * are needed while `stages` or `taus` is non-NULL (n_stages still reports the
 * count). */
hocResult_t hoc_topo_schedule(int G, const int* node_of, const int* sym, const uint64_t* C, uint64_t bw_nvlink,
                              uint64_t bw_rdma, uint64_t* T, uint64_t* stages, double* taus, int max_stages,
                              int* n_stages, double* total);

#ifdef __cplusplus
}
#endif

#endif /* HOC_SCHED_H */
