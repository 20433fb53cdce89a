// Two-domain stage scheduler (HOCCL section 3.4, Fig. 6, Eqs. 2-11,
// Algorithm 1).  Host only; see include/hoc_sched.h for the contract and the
// choices made where the algorithm leaves one open.
#include <algorithm>
#include <cstring>
#include <vector>

#include "hoc_sched.h"

namespace {

struct Cell {
  int u, v;
};

// Greedy contention-free matching over the cells with a positive value:
// largest value first, ties by (row, column); a cell is taken when its row
// and its column are both still free.
std::vector<Cell> greedy_matching(const std::vector<uint64_t>& val, const std::vector<Cell>& cells, int G) {
  std::vector<Cell> cand;
  for (const Cell& c : cells)
    if (val[size_t(c.u) * G + c.v] > 0) cand.push_back(c);
  std::sort(cand.begin(), cand.end(), [&](const Cell& a, const Cell& b) {
    const uint64_t x = val[size_t(a.u) * G + a.v], y = val[size_t(b.u) * G + b.v];
    if (x != y) return x > y;
    if (a.u != b.u) return a.u < b.u;
    return a.v < b.v;
  });
  std::vector<char> row(G, 0), col(G, 0);
  std::vector<Cell> out;
  for (const Cell& c : cand) {
    if (row[c.u] || col[c.v]) continue;
    row[c.u] = col[c.v] = 1;
    out.push_back(c);
  }
  return out;
}

struct Component {
  std::vector<Cell> cells;
  uint64_t weight;
};

}  // namespace

extern "C" hocResult_t hoc_topo_schedule(int G, const int* node_of, const int* sym, const uint64_t* C,
                                         uint64_t bw_nvlink, uint64_t bw_rdma, uint64_t* T_out, uint64_t* stages_out,
                                         double* taus_out, int max_stages, int* n_stages, double* total) {
  if (n_stages) *n_stages = 0;
  if (total) *total = 0.0;
  if (G < 1 || G > 64 || !node_of || !sym || !C || bw_nvlink == 0 || bw_rdma == 0 || max_stages < 0)
    return HOC_ERR_INVALID_ARG;
  for (int u = 0; u < G; ++u) {
    const int s = sym[u];
    if (s < 0 || s >= G || s == u || sym[s] != u || node_of[s] != node_of[u]) return HOC_ERR_INVALID_ARG;
    if (C[size_t(u) * G + u] != 0) return HOC_ERR_INVALID_ARG;
  }
  const size_t GG = size_t(G) * G;
  std::vector<Cell> inter, intra;
  for (int u = 0; u < G; ++u)
    for (int v = 0; v < G; ++v) {
      if (u == v) continue;
      (node_of[u] == node_of[v] ? intra : inter).push_back(Cell{u, v});
    }

  // Eqs. 2-4: T = C plus the forwarding copies on each (u, sym[u]) cell.
  std::vector<uint64_t> A(G, 0), B(G, 0);
  for (const Cell& c : inter) {
    A[c.u] += C[size_t(c.u) * G + c.v];
    B[c.v] += C[size_t(c.u) * G + c.v];
  }
  std::vector<uint64_t> T(C, C + GG);
  for (int u = 0; u < G; ++u) T[size_t(u) * G + sym[u]] += A[u] + B[sym[u]];
  if (T_out) memcpy(T_out, T.data(), GG * sizeof(uint64_t));

  // Step 2: native intra-node traffic of each NVLink domain peeled into matchings.
  std::vector<int> dom(node_of, node_of + G);
  std::sort(dom.begin(), dom.end());
  dom.erase(std::unique(dom.begin(), dom.end()), dom.end());
  std::vector<Component> comps;
  for (int d : dom) {
    std::vector<Cell> cells;
    for (const Cell& c : intra)
      if (node_of[c.u] == d) cells.push_back(c);
    std::vector<uint64_t> N(GG, 0);
    for (const Cell& c : cells) N[size_t(c.u) * G + c.v] = C[size_t(c.u) * G + c.v];
    for (;;) {
      std::vector<Cell> m = greedy_matching(N, cells, G);
      if (m.empty()) break;
      uint64_t w = UINT64_MAX;
      for (const Cell& c : m) w = std::min(w, N[size_t(c.u) * G + c.v]);
      for (const Cell& c : m) N[size_t(c.u) * G + c.v] -= w;
      comps.push_back(Component{m, w});
    }
  }

  // Steps 3-9: one stage per RDMA matching portion, NVLink slack filled.
  std::vector<uint64_t> R(GG, 0);
  for (const Cell& c : inter) R[size_t(c.u) * G + c.v] = C[size_t(c.u) * G + c.v];
  std::vector<std::vector<uint64_t>> stages;
  std::vector<double> taus;
  for (;;) {
    std::vector<Cell> m = greedy_matching(R, inter, G);
    if (m.empty()) break;
    uint64_t x = UINT64_MAX;
    for (const Cell& c : m) x = std::min(x, R[size_t(c.u) * G + c.v]);
    std::vector<uint64_t> S(GG, 0);
    for (const Cell& c : m) {
      S[size_t(c.u) * G + c.v] += x;
      R[size_t(c.u) * G + c.v] -= x;
      S[size_t(c.u) * G + sym[c.u]] += x;  // sender-side forwarding copy
      S[size_t(sym[c.v]) * G + c.v] += x;  // receiver-side forwarding copy
    }
    uint64_t l_nv = 0;
    for (const Cell& c : intra) l_nv = std::max(l_nv, S[size_t(c.u) * G + c.v]);
    uint64_t cap;
    double tau;
    if ((unsigned __int128)x * bw_nvlink >= (unsigned __int128)l_nv * bw_rdma) {  // RDMA-bound stage
      cap = uint64_t((unsigned __int128)x * bw_nvlink / bw_rdma);
      tau = double(x) / double(bw_rdma);
    } else {  // NVLink-bound stage
      cap = l_nv;
      tau = double(l_nv) / double(bw_nvlink);
    }
    for (Component& comp : comps) {
      if (comp.weight == 0) continue;
      uint64_t room = UINT64_MAX;
      for (const Cell& c : comp.cells) {
        const uint64_t used = S[size_t(c.u) * G + c.v];
        room = std::min(room, cap > used ? cap - used : 0);
      }
      const uint64_t a = std::min(comp.weight, room);
      if (a == 0) continue;
      for (const Cell& c : comp.cells) S[size_t(c.u) * G + c.v] += a;
      comp.weight -= a;
    }
    stages.push_back(std::move(S));
    taus.push_back(tau);
  }
  // Leftover native traffic: NVLink domains run in parallel, so each further
  // stage takes the next remaining matching of every domain.
  std::vector<std::vector<const Component*>> queue(dom.size());
  for (const Component& comp : comps) {
    if (comp.weight == 0) continue;
    const int d = int(std::lower_bound(dom.begin(), dom.end(), node_of[comp.cells[0].u]) - dom.begin());
    queue[d].push_back(&comp);
  }
  std::vector<size_t> head(dom.size(), 0);
  for (;;) {
    bool any = false;
    std::vector<uint64_t> S(GG, 0);
    uint64_t longest = 0;
    for (size_t d = 0; d < dom.size(); ++d) {
      if (head[d] >= queue[d].size()) continue;
      const Component* comp = queue[d][head[d]++];
      for (const Cell& c : comp->cells) S[size_t(c.u) * G + c.v] = comp->weight;
      longest = std::max(longest, comp->weight);
      any = true;
    }
    if (!any) break;
    stages.push_back(std::move(S));
    taus.push_back(double(longest) / double(bw_nvlink));
  }

  const int n = int(stages.size());
  if (n_stages) *n_stages = n;
  double sum = 0.0;
  for (double t : taus) sum += t;
  if (total) *total = sum;
  if ((stages_out || taus_out) && n > max_stages) return HOC_ERR_OOM;
  for (int s = 0; s < n; ++s) {
    if (stages_out) memcpy(stages_out + size_t(s) * GG, stages[s].data(), GG * sizeof(uint64_t));
    if (taus_out) taus_out[s] = taus[s];
  }
  return HOC_SUCCESS;
}
