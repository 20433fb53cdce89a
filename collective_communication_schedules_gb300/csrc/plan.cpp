// Collective scheduler (HOCCL section 3.4): chunking, ring order, pipeline
// edges, copy-queue striping, shift stages and flow-size-aware interleave.
#include "plan.h"

#include <algorithm>
#include <new>
#include <map>
#include <tuple>
#include <cstring>
#include <queue>

namespace hoc {

size_t dtype_bytes(int dtype) {
  switch (dtype) {
    case HOC_INT32:
    case HOC_FLOAT32: return 4;
    case HOC_BFLOAT16: return 2;
    case HOC_UINT8: return 1;
    default: return 0;
  }
}

int dtype_lanes(int dtype) { return dtype_bytes(dtype) ? int(16 / dtype_bytes(dtype)) : 0; }

void block_partition(size_t n, int k, std::vector<size_t>* sizes, std::vector<size_t>* offs) {
  sizes->assign(k, 0);
  offs->assign(k, 0);
  for (int r = 0; r < k; ++r) (*sizes)[r] = n / k + (size_t(r) < n % k ? 1 : 0);
  for (int r = 1; r < k; ++r) (*offs)[r] = (*offs)[r - 1] + (*sizes)[r - 1];
}

std::vector<std::pair<int, size_t>> interleave_chunks(const std::vector<size_t>& n, bool size_aware) {
  std::vector<std::pair<int, size_t>> out;
  size_t total = 0;
  for (size_t c : n) total += c;
  out.reserve(total);
  if (!size_aware) {
    for (size_t f = 0; f < n.size(); ++f)
      for (size_t j = 0; j < n[f]; ++j) out.emplace_back(int(f), j);
    return out;
  }
  // Min-heap on due time (j + 1) / n_f, compared exactly as (j+1)*n_g < (j'+1)*n_f.
  struct Head {
    int f;
    size_t j, nf;
  };
  auto later = [](const Head& a, const Head& b) {
    const unsigned __int128 x = (unsigned __int128)(a.j + 1) * b.nf;
    const unsigned __int128 y = (unsigned __int128)(b.j + 1) * a.nf;
    if (x != y) return x > y;
    return a.f > b.f;
  };
  std::priority_queue<Head, std::vector<Head>, decltype(later)> pq(later);
  for (size_t f = 0; f < n.size(); ++f)
    if (n[f]) pq.push({int(f), 0, n[f]});
  while (!pq.empty()) {
    Head h = pq.top();
    pq.pop();
    out.emplace_back(h.f, h.j);
    if (h.j + 1 < h.nf) pq.push({h.f, h.j + 1, h.nf});
  }
  return out;
}

std::string plan_key(const CallShape& s) {
  std::string key;
  auto put = [&key](const void* p, size_t n) { key.append(static_cast<const char*>(p), n); };
  put(&s.op, sizeof s.op);
  put(&s.k, sizeof s.k);
  put(&s.dtype, sizeof s.dtype);
  put(&s.count, sizeof s.count);
  put(&s.src_rank, sizeof s.src_rank);
  put(&s.dst_rank, sizeof s.dst_rank);
  put(&s.path, sizeof s.path);
  put(&s.chunk, sizeof s.chunk);
  const size_t nc = s.counts.size();
  put(&nc, sizeof nc);
  if (nc) put(s.counts.data(), nc * sizeof(size_t));
  const size_t ns = s.sdispls.size(), nr = s.rdispls.size();
  put(&ns, sizeof ns);
  if (ns) put(s.sdispls.data(), ns * sizeof(size_t));
  put(&nr, sizeof nr);
  if (nr) put(s.rdispls.data(), nr * sizeof(size_t));
  return key;
}

std::vector<std::vector<int>> source_groups(const std::vector<Move>& moves) {
  std::vector<std::vector<int>> groups;
  std::map<std::tuple<int, int, size_t, size_t>, size_t> open;  // source -> group still taking members
  for (size_t i = 0; i < moves.size(); ++i) {
    const Move& m = moves[i];
    const auto key = std::make_tuple(m.src_rank, m.src_buf, m.src_off, m.bytes);
    auto it = open.find(key);
    if (it != open.end() && groups[it->second].size() < size_t(kMaxRanks)) {
      groups[it->second].push_back(int(i));
    } else {
      open[key] = groups.size();
      groups.push_back({int(i)});
    }
  }
  return groups;
}

namespace {

size_t chunk_elems(size_t chunk_bytes, size_t b) {
  // whole kCopyAlignBytes units where the chunk holds one (so that chunks cut
  // from an aligned offset stay aligned), else 16-element multiples
  if (chunk_bytes >= kCopyAlignBytes) return chunk_bytes / kCopyAlignBytes * kCopyAlignBytes / b;
  size_t ce = chunk_bytes / b;
  ce -= ce % 16;
  return ce < 16 ? 16 : ce;
}

// Pieces of a move of about `chunk` bytes: cut on kCopyAlignBytes offsets of
// the destination (the first piece runs from the move's start to one chunk
// past the first such offset), a last piece under a quarter chunk merged into
// the one before.  (Copying the bytes before the first aligned offset as a
// piece of their own was tried for destinations not even 16-byte aligned:
// all-gathers gained, all-to-alls of single-piece flows lost, 0.416 -> 0.456
// ms.)  (offset into the move, bytes) each.
std::vector<std::pair<size_t, size_t>> move_pieces(size_t dst_off, size_t bytes, size_t chunk) {
  std::vector<std::pair<size_t, size_t>> v;
  if (bytes == 0) return v;
  const size_t head = (kCopyAlignBytes - dst_off % kCopyAlignBytes) % kCopyAlignBytes;
  size_t off = 0;
  size_t next = std::min(bytes, head + chunk);
  for (;;) {
    if (bytes - next < chunk / 4) next = bytes;
    v.emplace_back(off, next - off);
    if (next == bytes) break;
    off = next;
    next = std::min(bytes, off + chunk);
  }
  return v;
}

// Split `m` into its pieces (move_pieces).
void split_move(const Move& m, size_t chunk, std::vector<Move>* out) {
  for (const auto& pc : move_pieces(m.dst_off, m.bytes, chunk)) {
    Move c = m;
    c.src_off += pc.first;
    c.dst_off += pc.first;
    c.bytes = pc.second;
    out->push_back(c);
  }
}

void account(Plan* p) {
  p->bytes_exec = 0;
  p->kernels = 0;
  p->copies = 0;
  const size_t b = dtype_bytes(p->dtype);
  for (const Step& s : p->steps) {
    if (s.kind == kStepReduce || s.kind == kStepFused) {
      bool any = false;
      for (const ReduceSeg& g : s.segs) {
        const size_t outs = s.kind == kStepFused ? size_t(p->k) : 1;
        p->bytes_exec += (size_t(p->k) + outs) * g.elems * b;
        any = any || g.elems;
      }
      if (any) ++p->kernels;
    } else if (s.kind == kStepCopy) {
      size_t moved = 0;
      for (const Move& m : s.moves) moved += m.bytes;
      p->bytes_exec += 2 * moved;
      for (const Move& m : s.moves) p->copies += m.bytes ? 1 : 0;
    } else {  // TMA: a source shared by a group of moves is read once
      const auto groups = source_groups(s.moves);
      size_t written = 0, read = 0;
      for (const Move& m : s.moves) written += m.bytes;
      for (const auto& g : groups) read += s.moves[g[0]].bytes;
      p->bytes_exec += read + written;
      if (written) p->kernels += int((groups.size() + kMaxCopyJobs - 1) / kMaxCopyJobs);
    }
  }
  int streams = 1;
  for (const Step& s : p->steps) streams = std::max(streams, s.stream + 1);
  p->n_streams = streams;
}

// Host-side fault injection: corrupt the plan the way a broken scheduler or a
// lost DMA completion would, without touching memory outside the buffers.
void inject(const Cfg& cfg, Plan* p) {
  if (cfg.fault == kFaultWrongOrder) {
    for (Step& s : p->steps) s.waits.clear();
    return;
  }
  if (cfg.fault != kFaultDropChunk && cfg.fault != kFaultDupChunk) return;
  Move* first = nullptr;
  Step* last_step = nullptr;
  for (Step& s : p->steps) {
    if (s.kind != kStepCopy && s.kind != kStepTma) continue;
    for (Move& m : s.moves)
      if (!first && m.bytes) first = &m;
    if (!s.moves.empty()) last_step = &s;
  }
  if (!last_step || !first) return;
  if (cfg.fault == kFaultDropChunk) {
    last_step->moves.pop_back();
  } else {
    Move dup = last_step->moves.back();
    dup.dst_rank = first->dst_rank;
    dup.dst_buf = first->dst_buf;
    dup.dst_off = first->dst_off;
    dup.bytes = std::min(dup.bytes, first->bytes);
    if (dup.src_rank == first->dst_rank && dup.src_buf == dup.dst_buf && dup.src_off == dup.dst_off) return;
    last_step->moves.push_back(dup);
  }
}

int move_path(const Cfg& cfg) { return cfg.path == HOC_PATH_TMA ? HOC_PATH_TMA : HOC_PATH_CE; }

// Chunks of one flow set dealt round-robin over the copy streams (CE) or
// gathered into one bulk-copy launch (TMA).
// The largest copy of a chunk list (what the copy-queue count is chosen by).
size_t largest_copy(const std::vector<Move>& chunks) {
  size_t m = 0;
  for (const Move& c : chunks) m = std::max(m, c.bytes);
  return m;
}

void emit_moves(const Cfg& cfg, int path, const std::vector<Move>& chunks, int stage, const std::vector<int>& waits,
                bool record, Plan* p, std::vector<int>* step_ids, int queues) {
  if (chunks.empty()) return;
  if (path == HOC_PATH_TMA) {
    Step s;
    s.kind = kStepTma;
    s.stream = 1;
    s.stage = stage;
    s.moves = chunks;
    s.waits = waits;
    s.record = record;
    step_ids->push_back(int(p->steps.size()));
    p->steps.push_back(std::move(s));
    return;
  }
  const int n = std::max(1, queues);
  std::vector<Step> per(n);
  for (size_t i = 0; i < chunks.size(); ++i) per[i % n].moves.push_back(chunks[i]);
  for (int q = 0; q < n; ++q) {
    if (per[q].moves.empty()) continue;
    per[q].kind = kStepCopy;
    per[q].stream = 1 + q;
    per[q].stage = stage;
    per[q].waits = waits;
    per[q].record = record;
    step_ids->push_back(int(p->steps.size()));
    p->steps.push_back(std::move(per[q]));
  }
}

hocResult_t plan_allreduce(const Cfg& cfg, const CallShape& s, Plan* p) {
  const int k = s.k;
  const size_t b = dtype_bytes(s.dtype);
  std::vector<size_t> sz, off;
  block_partition(s.count, k, &sz, &off);
  p->bytes_min = 2 * size_t(k) * s.count * b;
  if (p->path == HOC_PATH_FUSED || k == 1) {
    Step st;
    st.kind = k == 1 ? kStepReduce : kStepFused;
    for (int r = 0; r < k; ++r)
      if (sz[r]) st.segs.push_back(ReduceSeg{off[r], sz[r], off[r], uint32_t(r), 0});
    p->steps.push_back(std::move(st));
    return HOC_SUCCESS;
  }
  const size_t ce = chunk_elems(allreduce_chunk(cfg, p->path, k), b);
  // Chunk boundaries inside a block sit on kCopyAlignBytes offsets of the
  // buffers: chunk 0 of owner r runs from the block's start to the first
  // aligned offset past it plus one chunk, the rest are whole chunks from
  // there.  Which rank owns an element (and so its fold order) is the
  // block's; only where the pipeline cuts it moves.
  const size_t ae = kCopyAlignBytes / b;
  std::vector<size_t> body(k);  // first aligned element of each block (clamped to its end)
  size_t nq = 1;
  for (int r = 0; r < k; ++r) {
    const size_t end = off[r] + sz[r];
    body[r] = std::min(end, (off[r] + ae - 1) / ae * ae);
    nq = std::max(nq, sz[r] ? std::max<size_t>(1, (end - body[r] + ce - 1) / ce) : size_t(1));
  }
  // chunk q of owner r: [*lo, *lo + *n); false if the block has no chunk q
  auto chunk_of = [&](int r, size_t q, size_t* lo, size_t* n) {
    const size_t end = off[r] + sz[r];
    const size_t a = q == 0 ? off[r] : body[r] + q * ce;
    if (sz[r] == 0 || a >= end) return false;
    *lo = a;
    *n = std::min(end, body[r] + (q + 1) * ce) - a;
    return true;
  };
  const int queues = copy_queues(cfg, std::min(ce, sz[0]) * b);
  std::vector<std::vector<int>> copy_steps(nq);
  for (size_t q = 0; q < nq; ++q) {
    Step red;
    red.kind = kStepReduce;
    red.stage = int(q);
    red.record = true;
    if (cfg.depth > 0 && q >= size_t(cfg.depth)) red.waits = copy_steps[q - cfg.depth];
    std::vector<Move> moves;
    for (int r = 0; r < k; ++r) {
      size_t lo, n;
      if (chunk_of(r, q, &lo, &n)) red.segs.push_back(ReduceSeg{lo, n, lo, uint32_t(r), 0});
    }
    // owner r's finished chunk goes to every other rank, shift by shift
    for (int t = 1; t < k; ++t)
      for (int r = 0; r < k; ++r) {
        size_t lo, n;
        if (!chunk_of(r, q, &lo, &n)) continue;
        const size_t byte_off = lo * b;
        moves.push_back(Move{r, (r + t) % k, HOC_BUF_RECV, HOC_BUF_RECV, byte_off, byte_off, n * b});
      }
    const int red_id = int(p->steps.size());
    p->steps.push_back(std::move(red));
    emit_moves(cfg, p->path, moves, int(q), {red_id}, cfg.depth > 0, p, &copy_steps[q], queues);
  }
  return HOC_SUCCESS;
}

hocResult_t plan_reduce_scatter(const Cfg&, const CallShape& s, Plan* p) {
  const int k = s.k;
  const size_t b = dtype_bytes(s.dtype);
  const size_t rc = s.count;
  Step st;
  st.kind = kStepReduce;
  for (int r = 0; r < k; ++r)
    if (rc) st.segs.push_back(ReduceSeg{size_t(r) * rc, rc, 0, uint32_t(r), 0});
  p->steps.push_back(std::move(st));
  p->bytes_min = (size_t(k) * k * rc + size_t(k) * rc) * b;
  return HOC_SUCCESS;
}

hocResult_t plan_allgather(const Cfg& cfg, const CallShape& s, Plan* p) {
  const int k = s.k;
  const size_t b = dtype_bytes(s.dtype);
  const size_t sc = s.count;
  std::vector<Move> chunks;
  for (int t = 0; t < k; ++t)
    for (int r = 0; r < k; ++r) {
      const int d = (r + t) % k;
      Move m{r, d, HOC_BUF_SEND, HOC_BUF_RECV, 0, size_t(r) * sc * b, sc * b};
      if (p->path == HOC_PATH_TMA) chunks.push_back(m);
      else split_move(m, chunk_for(cfg, HOC_PATH_CE), &chunks);
    }
  std::vector<int> ids;
  emit_moves(cfg, p->path, chunks, 0, {}, false, p, &ids, copy_queues(cfg, largest_copy(chunks)));
  if (p->path == HOC_PATH_TMA && !p->steps.empty()) p->steps.back().stream = 0;
  p->bytes_min = (size_t(k) * sc + size_t(k) * k * sc) * b;
  return HOC_SUCCESS;
}

hocResult_t plan_alltoall(const Cfg& cfg, const CallShape& s, Plan* p) {
  const int k = s.k;
  const size_t b = dtype_bytes(s.dtype);
  auto cnt = [&](int src, int dst) -> size_t {
    return s.counts.empty() ? s.count : s.counts[size_t(src) * k + dst];
  };
  // default displacements: prefix sums in rank order
  std::vector<size_t> sd(size_t(k) * k), rd(size_t(k) * k);
  for (int a = 0; a < k; ++a)
    for (int c = 0; c < k; ++c) {
      sd[size_t(a) * k + c] = s.sdispls.empty() ? (c ? sd[size_t(a) * k + c - 1] + cnt(a, c - 1) : 0)
                                                : s.sdispls[size_t(a) * k + c];
    }
  for (int d = 0; d < k; ++d)
    for (int a = 0; a < k; ++a) {
      rd[size_t(d) * k + a] = s.rdispls.empty() ? (a ? rd[size_t(d) * k + a - 1] + cnt(a - 1, d) : 0)
                                                : s.rdispls[size_t(d) * k + a];
    }
  size_t total = 0;
  for (int a = 0; a < k; ++a)
    for (int d = 0; d < k; ++d) total += cnt(a, d);
  p->bytes_min = 2 * total * b;
  if (p->path == HOC_PATH_TMA) {
    std::vector<Move> all;
    for (int st = 0; st < k; ++st)
      for (int u = 0; u < k; ++u) {
        const int v = (u + st) % k;
        const size_t n = cnt(u, v) * b;
        if (n) all.push_back(Move{u, v, HOC_BUF_SEND, HOC_BUF_RECV, sd[size_t(u) * k + v] * b, rd[size_t(v) * k + u] * b, n});
      }
    std::vector<int> ids;
    emit_moves(cfg, HOC_PATH_TMA, all, 0, {}, false, p, &ids, 1);
    if (!p->steps.empty()) p->steps.back().stream = 0;
    return HOC_SUCCESS;
  }
  // Shift stages (Eq. 6-8 with one domain): stage st holds flows u -> u+st.
  const size_t cb = chunk_for(cfg, HOC_PATH_CE);
  size_t biggest = 0;
  for (int a = 0; a < k; ++a)
    for (int d = 0; d < k; ++d) biggest = std::max(biggest, std::min(cb, cnt(a, d) * b));
  const int queues = copy_queues(cfg, biggest);
  std::vector<int> prev;
  for (int st = 0; st < k; ++st) {
    std::vector<Move> flows;
    std::vector<std::vector<std::pair<size_t, size_t>>> pieces;
    std::vector<size_t> nchunks;
    for (int u = 0; u < k; ++u) {
      const int v = (u + st) % k;
      const size_t n = cnt(u, v) * b;
      flows.push_back(Move{u, v, HOC_BUF_SEND, HOC_BUF_RECV, sd[size_t(u) * k + v] * b, rd[size_t(v) * k + u] * b, n});
      pieces.push_back(move_pieces(flows.back().dst_off, n, cb));
      nchunks.push_back(pieces.back().size());
    }
    std::vector<Move> chunks;
    for (const auto& fc : interleave_chunks(nchunks, cfg.a2a_interleave != 0)) {
      const Move& f = flows[fc.first];
      const auto& pc = pieces[fc.first][fc.second];
      chunks.push_back(Move{f.src_rank, f.dst_rank, f.src_buf, f.dst_buf, f.src_off + pc.first, f.dst_off + pc.first,
                            pc.second});
    }
    std::vector<int> ids;
    emit_moves(cfg, HOC_PATH_CE, chunks, st, cfg.a2a_stage_sync ? prev : std::vector<int>{}, cfg.a2a_stage_sync != 0,
               p, &ids, queues);
    if (!ids.empty()) prev = ids;
  }
  return HOC_SUCCESS;
}

hocResult_t plan_sendrecv(const Cfg& cfg, const CallShape& s, Plan* p) {
  const size_t bytes = s.count * dtype_bytes(s.dtype);
  Move m{s.src_rank, s.dst_rank, HOC_BUF_SEND, HOC_BUF_RECV, 0, 0, bytes};
  std::vector<Move> chunks;
  if (p->path == HOC_PATH_TMA || bytes <= kSendrecvStripeBytes) chunks.push_back(m);
  else split_move(m, chunk_for(cfg, HOC_PATH_CE), &chunks);
  std::vector<int> ids;
  emit_moves(cfg, p->path, chunks, 0, {}, false, p, &ids, copy_queues(cfg, largest_copy(chunks)));
  if (p->path == HOC_PATH_TMA && !p->steps.empty()) p->steps.back().stream = 0;
  p->bytes_min = 2 * bytes;
  return HOC_SUCCESS;
}

// The spans a call names stay within kMaxSpanBytes, and the largest one
// within kMaxChunksPerSpan chunks.  Every count is checked on its own before
// any sum, so no sum can wrap.
hocResult_t check_sizes(const Cfg& cfg, const CallShape& s) {
  const uint64_t b = dtype_bytes(s.dtype);
  const uint64_t lim = kMaxSpanBytes / b;  // elements in the largest span
  const uint64_t k = uint64_t(s.k);
  auto too_big = [] {
    set_error_detail("a rank's buffer span exceeds 2^40 bytes");
    return HOC_ERR_INVALID_ARG;
  };
  uint64_t span = 0;  // bytes of the largest rank buffer span
  switch (s.op) {
    case HOC_OP_ALLREDUCE:
    case HOC_OP_SENDRECV:
      if (s.count > lim) return too_big();
      span = s.count * b;
      break;
    case HOC_OP_REDUCE_SCATTER:
    case HOC_OP_ALLGATHER:
      if (s.count > lim / k) return too_big();
      span = s.count * k * b;
      break;
    case HOC_OP_ALLTOALL: {
      if (s.counts.empty()) {
        if (s.count > lim / k) return too_big();
        span = s.count * k * b;
        break;
      }
      if (s.counts.size() != k * k || (!s.sdispls.empty() && s.sdispls.size() != k * k) ||
          (!s.rdispls.empty() && s.rdispls.size() != k * k))
        return HOC_ERR_INVALID_ARG;
      std::vector<uint64_t> col(k, 0);
      for (uint64_t a = 0; a < k; ++a) {
        uint64_t row = 0;
        for (uint64_t d = 0; d < k; ++d) {
          const uint64_t c = s.counts[a * k + d];
          if (c > lim) return too_big();
          if (!s.sdispls.empty() && (s.sdispls[a * k + d] > lim || s.sdispls[a * k + d] + c > lim)) return too_big();
          if (!s.rdispls.empty() && (s.rdispls[d * k + a] > lim || s.rdispls[d * k + a] + c > lim)) return too_big();
          row += c;
          col[d] += c;
        }
        if (row > lim) return too_big();
        span = std::max(span, row * b);
      }
      for (uint64_t c : col) {
        if (c > lim) return too_big();
        span = std::max(span, c * b);
      }
      break;
    }
    default: return HOC_ERR_INVALID_ARG;
  }
  const uint64_t chunk =
      cfg.chunk_bytes ? cfg.chunk_bytes : std::min(std::min(kAutoChunkCe, kAutoChunkTma), kArChunkMinBytes);
  if (span / chunk > kMaxChunksPerSpan) {
    set_error_detail("chunk_bytes too small for this size: more than 2^24 chunks per rank buffer");
    return HOC_ERR_INVALID_ARG;
  }
  return HOC_SUCCESS;
}

hocResult_t build_plan_checked(const Cfg& base, const CallShape& s, Plan* p);

}  // namespace

hocResult_t build_plan(const Cfg& base, const CallShape& s, Plan* p) {
  try {
    return build_plan_checked(base, s, p);
  } catch (const std::bad_alloc&) {
    *p = Plan();
    set_error_detail("out of host memory while building the plan");
    return HOC_ERR_OOM;
  }
}

namespace {

hocResult_t build_plan_checked(const Cfg& base, const CallShape& s, Plan* p) {
  Cfg cfg = base;
  if (s.chunk) cfg.chunk_bytes = s.chunk;
  *p = Plan();
  p->op = s.op;
  p->k = s.k;
  p->dtype = s.dtype;
  p->count = s.count;
  if (s.k < 1 || s.k > kMaxRanks || dtype_bytes(s.dtype) == 0) return HOC_ERR_INVALID_ARG;
  if ((cfg.chunk_bytes != 0 && cfg.chunk_bytes < 256) || cfg.n_copy < 1 || cfg.n_copy > 16) return HOC_ERR_INVALID_ARG;
  hocResult_t r = check_sizes(cfg, s);
  if (r != HOC_SUCCESS) return r;
  switch (s.op) {
    case HOC_OP_ALLREDUCE:
      if (s.dtype == HOC_UINT8) return HOC_ERR_UNSUPPORTED;
      // AUTO: the fused kernel with the whole GPU; under an SM budget the copy
      // engines take the moves, so the few SMs only reduce.
      p->path = s.path >= 0 ? s.path
                            : (cfg.path != HOC_PATH_AUTO ? cfg.path
                                                         : (cfg.reduce_max_sms > 0 ? HOC_PATH_CE : HOC_PATH_FUSED));
      if (p->path < HOC_PATH_CE || p->path > HOC_PATH_FUSED) return HOC_ERR_INVALID_ARG;
      r = plan_allreduce(cfg, s, p);
      break;
    case HOC_OP_REDUCE_SCATTER:
      if (s.dtype == HOC_UINT8) return HOC_ERR_UNSUPPORTED;
      p->path = HOC_PATH_FUSED;  // one reduce kernel; no moves
      r = plan_reduce_scatter(cfg, s, p);
      break;
    case HOC_OP_ALLGATHER:
      p->path = move_path(cfg);
      r = plan_allgather(cfg, s, p);
      break;
    case HOC_OP_ALLTOALL:
      p->path = move_path(cfg);
      r = plan_alltoall(cfg, s, p);
      break;
    case HOC_OP_SENDRECV:
      p->path = move_path(cfg);
      r = plan_sendrecv(cfg, s, p);
      break;
    default: return HOC_ERR_INVALID_ARG;
  }
  if (r != HOC_SUCCESS) return r;
  inject(cfg, p);
  // drop empty steps, remapping wait indices
  std::vector<int> remap(p->steps.size(), -1);
  std::vector<Step> kept;
  for (size_t i = 0; i < p->steps.size(); ++i) {
    Step& st = p->steps[i];
    const bool empty = (st.kind == kStepReduce || st.kind == kStepFused) ? st.segs.empty() : st.moves.empty();
    if (empty) continue;
    remap[i] = int(kept.size());
    kept.push_back(std::move(st));
  }
  for (Step& st : kept) {
    std::vector<int> w;
    for (int x : st.waits)
      if (x >= 0 && remap[x] >= 0) w.push_back(remap[x]);
    st.waits = w;
  }
  p->steps = std::move(kept);
  // A plan that uses a single internal stream runs on the caller's stream instead (no fork/join).
  int used = -1;
  bool single = true;
  for (const Step& st : p->steps) {
    if (used < 0) used = st.stream;
    else if (st.stream != used) single = false;
  }
  if (single && used > 0)
    for (Step& st : p->steps) st.stream = 0;
  for (Step& st : p->steps)
    for (int w : st.waits) p->steps[w].record = true;
  account(p);
  return HOC_SUCCESS;
}

}  // namespace

}  // namespace hoc
