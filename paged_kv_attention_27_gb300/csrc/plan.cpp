// Host planner: validation, split-KV decisions, work list and workspace
// sizing. Pure host code (no CUDA calls), so it runs and is tested on a
// machine without a GPU.
//
// Scheduling by sequence length follows the idea of "FlashInfer Attention
// Kernel optimisation analysis", section 2.2 (dynamic load balancing by
// sequence length) and "FlashInfer kernel library deep-dive", section
// "load-balanced scheduling": long KV is cut into chunks so that no CTA
// carries far more than the average load, and the largest items launch
// first (longest-processing-time order), which bounds the tail.
#include <algorithm>
#include <cstring>

#include "fi_internal.h"

namespace fi {

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

}  // namespace

fi_status build_plan(int32_t mode, int32_t batch, const int32_t* qo_indptr,
                     const int32_t* page_indptr, const int32_t* last_page_len,
                     int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t page_size, int32_t causal, const fi_plan_options* options,
                     int32_t num_sms, Plan* out) {
  if (!out) return FI_ERR_INVALID_ARG;
  const fi_plan_options opt = options ? *options : fi_plan_options FI_PLAN_OPTIONS_DEFAULT;
  if (opt.window_left < -1) return FI_ERR_INVALID_ARG;
  if (opt.dtype != FI_DTYPE_BF16 && opt.dtype != FI_DTYPE_FP16) return FI_ERR_INVALID_ARG;
  const int32_t kv_dtype = opt.kv_dtype < 0 ? opt.dtype : opt.kv_dtype;
  if (kv_dtype != opt.dtype && kv_dtype != FI_DTYPE_E4M3) return FI_ERR_INVALID_ARG;
  if (mode != FI_MODE_DECODE && mode != FI_MODE_PREFILL) return FI_ERR_INVALID_ARG;
  if (batch < 0 || num_sms <= 0) return FI_ERR_INVALID_ARG;
  if (num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0)
    return FI_ERR_INVALID_ARG;
  if (num_qo_heads % num_kv_heads != 0) return FI_ERR_INVALID_ARG;
  if (batch > 0 && (!page_indptr || !last_page_len)) return FI_ERR_INVALID_ARG;
  if (mode == FI_MODE_DECODE && qo_indptr) return FI_ERR_INVALID_ARG;
  if (mode == FI_MODE_PREFILL && batch > 0 && !qo_indptr) return FI_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return FI_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32) return FI_ERR_UNSUPPORTED;
  const int g = num_qo_heads / num_kv_heads;
  if (!supported_group(g)) return FI_ERR_UNSUPPORTED;

  Plan p;
  p.mode = mode;
  p.batch = batch;
  p.num_qo_heads = num_qo_heads;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.page_size = page_size;
  p.causal = (mode == FI_MODE_PREFILL) ? (causal ? 1 : 0) : 0;
  p.num_sms = num_sms;
  p.window_left = opt.window_left;
  p.dtype = opt.dtype;
  p.kv_dtype = kv_dtype;
  // an FP8 cache is read by the decode kernel only
  if (kv_dtype == FI_DTYPE_E4M3 && mode != FI_MODE_DECODE) return FI_ERR_UNSUPPORTED;

  // ---- validate the page table and the query packing; kv_len per request
  std::vector<int64_t> kv_len(batch), qo_len(batch), qo_start(batch);
  if (batch > 0 && page_indptr[0] < 0) return FI_ERR_INVALID_ARG;
  if (mode == FI_MODE_PREFILL && batch > 0 && qo_indptr[0] != 0) return FI_ERR_INVALID_ARG;
  int64_t total_q = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t np = int64_t(page_indptr[b + 1]) - page_indptr[b];
    if (np < 0) return FI_ERR_INVALID_ARG;
    if (np > 0) {
      if (last_page_len[b] < 1 || last_page_len[b] > page_size) return FI_ERR_INVALID_ARG;
      kv_len[b] = (np - 1) * page_size + last_page_len[b];
    } else {
      if (last_page_len[b] < 0 || last_page_len[b] > page_size) return FI_ERR_INVALID_ARG;
      kv_len[b] = 0;
    }
    if (kv_len[b] > INT32_MAX / 2) return FI_ERR_INVALID_ARG;
    if (mode == FI_MODE_PREFILL) {
      qo_len[b] = int64_t(qo_indptr[b + 1]) - qo_indptr[b];
      if (qo_len[b] < 0) return FI_ERR_INVALID_ARG;
      if (p.causal && qo_len[b] > kv_len[b]) return FI_ERR_INVALID_ARG;
      qo_start[b] = qo_indptr[b];
    } else {
      qo_len[b] = 1;
      qo_start[b] = b;
    }
    total_q += qo_len[b];
    p.total_kv += kv_len[b];
  }
  if (total_q > INT32_MAX) return FI_ERR_INVALID_ARG;
  p.total_q = total_q;

  // prefill-kernel tiles of the shared-prefix level: 128 M rows = (128 / g
  // rows of q) x (the g query heads of one kv head), so that every K/V tile
  // serves the whole group. (Ordinary prefill keeps 128 rows of one query
  // head per tile: packing measured slower on long causal prefill.)
  const int64_t rows_per_tile = kPrefillTileM / g;

  // ---- shared-prefix groups (decode plans): group g's requests share their
  //      first prefix_pages[g] pages; the prefix is attended once per group
  //      and each request's decode work starts after it
  const int G = opt.num_prefix_groups;
  std::vector<int64_t> prefix_tokens(batch, 0);
  if (G < 0) return FI_ERR_INVALID_ARG;
  if (G > 0) {
    if (!opt.prefix_group_indptr || !opt.prefix_pages) return FI_ERR_INVALID_ARG;
    if (mode != FI_MODE_DECODE || kv_dtype == FI_DTYPE_E4M3 || opt.window_left >= 0)
      return FI_ERR_UNSUPPORTED;
    const int32_t* gi = opt.prefix_group_indptr;
    if (gi[0] < 0 || gi[G] > batch) return FI_ERR_INVALID_ARG;
    for (int g = 0; g < G; ++g) {
      if (gi[g + 1] < gi[g]) return FI_ERR_INVALID_ARG;
      const int64_t pages = opt.prefix_pages[g];
      if (pages < 1) return FI_ERR_INVALID_ARG;
      for (int b = gi[g]; b < gi[g + 1]; ++b) {
        const int64_t np = int64_t(page_indptr[b + 1]) - page_indptr[b];
        // the prefix is made of full pages of every request in the group
        if (np < pages || (np == pages && last_page_len[b] != page_size))
          return FI_ERR_INVALID_ARG;
        prefix_tokens[b] = pages * page_size;
      }
    }
  }

  // ---- the keys a row may see: [first_key, ...). A left window moves the
  //      start; the row at key position pos keeps keys t >= pos - window_left.
  //      (For decode work of a shared-prefix request: the first key after
  //      the prefix, which is attended separately.)
  auto first_key = [&](int b, int64_t row) -> int64_t {
    if (prefix_tokens[b] > 0) return prefix_tokens[b];
    if (p.window_left < 0) return 0;
    return std::max<int64_t>(0, kv_len[b] - qo_len[b] + row - p.window_left);
  };
  // Each group's prefix is cut into chunks so that its items fill about two
  // waves of the GPU (the prefix can be long and the group small); chunk c
  // of group g writes one state per row of the group, in slots
  // pslot[g] + c * rows(g) + (row - first row). The decode merge adds them.
  std::vector<int64_t> pchunk(std::max(G, 0), 0), pn(std::max(G, 0), 0), prow0(std::max(G, 0), 0),
      pnrow(std::max(G, 0), 0), pslot(std::max(G, 0), 0);
  std::vector<int32_t> group_of(batch, -1);
  for (int g = 0; g < G; ++g) {
    const int b0 = opt.prefix_group_indptr[g], b1 = opt.prefix_group_indptr[g + 1];
    if (b1 <= b0) continue;
    for (int b = b0; b < b1; ++b) group_of[b] = g;
    const int64_t Lp = int64_t(opt.prefix_pages[g]) * page_size;
    prow0[g] = qo_start[b0];
    pnrow[g] = qo_start[b1 - 1] + 1 - prow0[g];
    const int64_t per_chunk = ceil_div(pnrow[g], rows_per_tile) * num_kv_heads;   // items
    const int64_t want = std::max<int64_t>(1, ceil_div(int64_t(num_sms) * 2, per_chunk));
    const int64_t n = std::min<int64_t>(want, std::max<int64_t>(1, Lp / 1024));
    pchunk[g] = ceil_div(ceil_div(Lp, n), 128) * 128;   // whole KV tiles
    pn[g] = ceil_div(Lp, pchunk[g]);
    pslot[g] = p.num_slots;
    p.num_slots += int32_t(pn[g] * pnrow[g]);
  }

  // ---- decode work: every request with exactly one query row. Chunks start
  //      on page boundaries from the page holding the first visible key.
  const int tile = decode_tile_tokens(head_dim);
  std::vector<int> dec;
  int64_t dec_tiles = 0;
  for (int b = 0; b < batch; ++b) {
    if (qo_len[b] == 1) {
      dec.push_back(b);
      const int64_t s0 = first_key(b, 0) / page_size * page_size;
      dec_tiles += std::max<int64_t>(1, ceil_div(kv_len[b] - s0, tile)) * num_kv_heads;
    }
  }
  if (!dec.empty()) {
    // Aim for ~4 items per resident decode CTA (2 per SM), so that the
    // largest item is a small fraction of one CTA's share, but never cut
    // chunks below 512 tokens (per-CTA setup would dominate). (The mixed
    // kernel measured slowest with finer chunks: 1.745 ms per call at this
    // target, 1.770 at twice it, 1.848 at four times.)
    const int64_t target = int64_t(num_sms) * 2 * 4;
    const int64_t min_chunk_tiles = std::max<int64_t>(1, 512 / tile);
    const int64_t chunk_tiles = std::max(min_chunk_tiles, ceil_div(dec_tiles, target));
    const int64_t chunk = chunk_tiles * tile;  // a multiple of the page size
    p.chunk_tokens = int32_t(std::min<int64_t>(chunk, INT32_MAX));
    // Every kv head of a (request, chunk) gets an item of the same length,
    // so the longest-first order is found by sorting the (request, chunk)
    // groups, not the items.
    struct Group { int64_t len; int32_t b, c; };
    std::vector<Group> groups;
    std::vector<int64_t> w0s(batch), s0s(batch);
    std::vector<int32_t> slot_base(batch, -1), merge_of(batch, -1);
    for (int b : dec) {
      const int64_t w0 = first_key(b, 0);
      const int64_t s0 = w0 / page_size * page_size;
      w0s[b] = w0;
      s0s[b] = s0;
      const int64_t n_chunks = std::max<int64_t>(1, ceil_div(kv_len[b] - s0, chunk));
      // split requests, and every request with a shared prefix, write
      // partial states that the decode kernel merges (plus the prefix state)
      const bool prefixed = prefix_tokens[b] > 0;
      if (n_chunks > 1 || prefixed) {
        merge_of[b] = int32_t(p.merges.size());
        slot_base[b] = p.num_slots;
        p.num_slots += int32_t(n_chunks);
        p.num_split += n_chunks > 1 ? 1 : 0;
        MergeTask mt{int32_t(qo_start[b]), slot_base[b], int32_t(n_chunks), -1, 0, 0, {0, 0}};
        if (prefixed) {
          const int g = group_of[b];
          mt.extra_slot = int32_t(pslot[g] + (qo_start[b] - prow0[g]));
          mt.n_extra = int32_t(pn[g]);
          mt.extra_stride = int32_t(pnrow[g]);
        }
        p.merges.push_back(mt);
      }
      for (int64_t c = 0; c < n_chunks; ++c) {
        const int64_t t0 = s0 + c * chunk;
        const int64_t t1 = std::min<int64_t>(kv_len[b], t0 + chunk);
        groups.push_back(Group{std::max<int64_t>(0, t1 - (c == 0 ? w0 : t0)), b, int32_t(c)});
      }
    }
    std::sort(groups.begin(), groups.end(), [](const Group& x, const Group& y) {
      if (x.len != y.len) return x.len > y.len;
      return x.b != y.b ? x.b < y.b : x.c < y.c;
    });
    // sized once and written through a pointer (a push_back per item cost
    // more than the rest of the plan together)
    p.decode_items.resize(groups.size() * size_t(num_kv_heads));
    WorkItem* dst = p.decode_items.data();
    for (const Group& g : groups) {
      const int b = g.b;
      const int64_t t0 = s0s[b] + int64_t(g.c) * chunk;   // page-aligned start of the chunk
      const int64_t t1 = std::min<int64_t>(kv_len[b], t0 + chunk);
      WorkItem w;
      w.req = b;
      w.page_begin = int32_t(page_indptr[b] + t0 / page_size);
      w.n_pages = int32_t(t1 > t0 ? ceil_div(t1 - t0, page_size) : 0);
      w.tok_begin = int32_t(g.c == 0 ? w0s[b] : t0);     // first visible key
      w.tok_end = int32_t(std::max(t0, t1));
      w.slot = slot_base[b] >= 0 ? slot_base[b] + g.c : -1;
      w.q_row = int32_t(qo_start[b]);
      w.merge = merge_of[b];
      for (int kh = 0; kh < num_kv_heads; ++kh) {
        w.head = kh;
        *dst++ = w;
      }
    }
  }

  // ---- shared-prefix work: per group, the group's rows of q (one query
  //      kv head per item, tiles of rows_per_tile rows) against the prefix, on
  //      the prefill kernel. Virtual request 2g describes group g to it:
  //      rows [first, last) of q, prefix_pages full pages, not causal.
  if (G > 0) {
    p.num_prefix_groups = G;
    p.prefix_tables.assign(size_t(6) * G, 0);
    int32_t* vq = p.prefix_tables.data();          // qo_indptr   [2G]
    int32_t* vp = vq + 2 * G;                      // page_indptr [2G]
    int32_t* vl = vq + 4 * G;                      // last_page_len [2G]
    struct PTile { int64_t len; int32_t g, c, r0; };
    std::vector<PTile> ptiles;
    for (int g = 0; g < G; ++g) {
      vq[2 * g] = int32_t(prow0[g]);
      vq[2 * g + 1] = int32_t(prow0[g] + pnrow[g]);
      vp[2 * g] = 0;
      vp[2 * g + 1] = opt.prefix_pages[g];
      vl[2 * g] = page_size;
      const int64_t Lp = int64_t(opt.prefix_pages[g]) * page_size;
      for (int64_t c = 0; c < pn[g]; ++c)
        for (int64_t r0 = prow0[g]; r0 < prow0[g] + pnrow[g]; r0 += rows_per_tile)
          ptiles.push_back(PTile{std::min(Lp, (c + 1) * pchunk[g]) - c * pchunk[g], g,
                                 int32_t(c), int32_t(r0)});
    }
    std::stable_sort(ptiles.begin(), ptiles.end(),
                     [](const PTile& x, const PTile& y) { return x.len > y.len; });
    p.prefix_items.resize(ptiles.size() * size_t(num_kv_heads));
    WorkItem* dst = p.prefix_items.data();
    for (const PTile& t : ptiles) {
      const int64_t k0 = int64_t(t.c) * pchunk[t.g];
      WorkItem w;
      w.req = 2 * t.g;
      // the group's first request holds the shared pages
      w.page_begin = int32_t(page_indptr[opt.prefix_group_indptr[t.g]] + k0 / page_size);
      w.n_pages = int32_t(ceil_div(t.len, page_size));
      w.tok_begin = int32_t(k0);
      w.tok_end = int32_t(k0 + t.len);
      w.slot = int32_t(pslot[t.g] + int64_t(t.c) * pnrow[t.g] - prow0[t.g]);
      w.q_row = t.r0;
      w.merge = -1;
      for (int kh = 0; kh < num_kv_heads; ++kh) {
        w.head = kh;
        *dst++ = w;
      }
    }
  }

  // ---- prefill work: requests with two or more query rows, one item per
  //      (query tile of kPrefillTileM rows, query head); the tiles are
  //      ordered longest first, the heads of a tile stay together, in head
  //      order (the two-tile kernel runs items 2p and 2p + 1 in one CTA)
  struct Tile { int64_t len, kv_begin, kv_end; int32_t b, qt; };
  std::vector<Tile> tiles;
  for (int b = 0; b < batch; ++b) {
    if (qo_len[b] < 2) continue;
    const int64_t n_qt = ceil_div(qo_len[b], kPrefillTileM);
    for (int64_t qt = 0; qt < n_qt; ++qt) {
      const int64_t r0 = qt * kPrefillTileM;
      const int64_t r_last = std::min<int64_t>(qo_len[b], r0 + kPrefillTileM) - 1;
      int64_t kv_end = kv_len[b];
      if (p.causal) kv_end = std::min<int64_t>(kv_len[b], kv_len[b] - qo_len[b] + r_last + 1);
      // the tile's first row has the smallest window start; tiles of keys
      // begin on the page that holds it
      const int64_t kv_begin = std::min(kv_end, first_key(b, r0)) / page_size * page_size;
      tiles.push_back(Tile{kv_end - kv_begin, kv_begin, kv_end, b, int32_t(qt)});
    }
  }
  std::sort(tiles.begin(), tiles.end(), [](const Tile& x, const Tile& y) {
    if (x.len != y.len) return x.len > y.len;
    return x.b != y.b ? x.b < y.b : x.qt < y.qt;
  });

  // ---- KV split of prefill tiles when the launch has under two waves of
  //      work units (a CTA's unit: a tile with one head, or with a head pair
  //      on the two-tile kernel). Long tiles are then cut into pieces of
  //      whole KV tiles, so that more SMs share the longest ones ("FlashInfer
  //      Attention Kernel optimisation analysis", section 2.2: balance the
  //      load by sequence length); each piece writes fp32 states (O / l and
  //      lse per row and head) and one merge launch combines a row's pieces
  //      by log-sum-exp. The piece count k of the longest tile minimises
  //      ceil(units * k / SMs) * (tiles / k + c0), the finish time of units
  //      of that length handed out in rounds, with c0 = kSplitPieceCost KV
  //      tiles per piece, and is taken only if that beats the whole tiles'
  //      estimate by the margin kSplitMaxRatio; shorter tiles are cut at the
  //      same length. Only a longest tile of kMinSplitTiles KV tiles or more
  //      is worth a merge launch, and plans with decode rows (the mixed
  //      kernel, concurrent decode) are not split.
  struct Piece { int64_t len, kv_begin, kv_end; int32_t b, qt, slot, k; };
  std::vector<Piece> pieces;
  pieces.reserve(tiles.size());
  {
    const int64_t kv_tile = prefill_kv_tile(head_dim);
    const int64_t heads_per_unit = (head_dim <= 128 && g % 2 == 0) ? 2 : 1;
    const int64_t units = int64_t(tiles.size()) * (num_qo_heads / heads_per_unit);
    int64_t split_len = 0;   // keys per piece (whole KV tiles); 0: no split
    if (dec.empty() && !tiles.empty() && units < 2 * int64_t(num_sms)) {
      const int64_t max_tiles = ceil_div(tiles[0].len, kv_tile);
      int64_t best_k = 1;
      if (max_tiles < kMinSplitTiles) best_k = 0;   // (no candidate below)
      const double whole = double(ceil_div(units, num_sms)) * double(max_tiles + kSplitPieceCost);
      double best = whole * kSplitMaxRatio;          // a split must beat this
      for (int64_t k = 2; best_k > 0 && k <= kMaxPrefillPieces && max_tiles >= 2 * k; ++k) {
        const double f = double(ceil_div(units * k, num_sms)) *
                         (double(max_tiles) / double(k) + double(kSplitPieceCost));
        if (f < best) {
          best = f;
          best_k = k;
        }
      }
      if (best_k > 1) split_len = ceil_div(max_tiles, best_k) * kv_tile;
    }
    for (const Tile& t : tiles) {
      const int64_t k = split_len > 0 ? std::max<int64_t>(1, ceil_div(t.len, split_len)) : 1;
      if (k == 1) {
        pieces.push_back(Piece{t.len, t.kv_begin, t.kv_end, t.b, t.qt, -1, -1});
        continue;
      }
      // slots of the tile's rows: row r, piece j -> slot s0 + r * k + j
      const int64_t rows = std::min<int64_t>(kPrefillTileM, qo_len[t.b] - int64_t(t.qt) * kPrefillTileM);
      const int64_t s0 = p.num_slots;
      p.num_slots += int32_t(rows * k);
      for (int64_t r = 0; r < rows; ++r) {
        MergeTask mt{int32_t(qo_start[t.b] + int64_t(t.qt) * kPrefillTileM + r),
                     int32_t(s0 + r * k), int32_t(k), -1, 0, 0, {0, 0}};
        p.prefill_merges.push_back(mt);
      }
      for (int64_t j = 0; j < k; ++j) {
        const int64_t b0 = t.kv_begin + j * split_len;
        const int64_t b1 = std::min(t.kv_end, b0 + split_len);
        pieces.push_back(Piece{b1 - b0, b0, b1, t.b, t.qt, int32_t(s0 + j), int32_t(k)});
      }
    }
    std::stable_sort(pieces.begin(), pieces.end(),
                     [](const Piece& x, const Piece& y) { return x.len > y.len; });
  }
  p.prefill_items.resize(pieces.size() * size_t(num_qo_heads));
  WorkItem* pdst = p.prefill_items.data();
  for (const Piece& t : pieces) {
    WorkItem w;
    w.req = t.b;
    w.page_begin = int32_t(page_indptr[t.b] + t.kv_begin / page_size);
    w.n_pages = int32_t(ceil_div(t.kv_end - t.kv_begin, page_size));
    w.tok_begin = int32_t(t.kv_begin);
    w.tok_end = int32_t(t.kv_end);
    w.slot = t.slot;   // a piece: its state of row r at slot + r * merge
    w.q_row = int32_t(qo_start[t.b] + int64_t(t.qt) * kPrefillTileM);
    w.merge = t.k;     // a piece: the tile's piece count; else -1
    for (int h = 0; h < num_qo_heads; ++h) {
      w.head = h;
      *pdst++ = w;
    }
  }

  // ---- workspace: header | decode items | prefill items | prefix items |
  //      prefix tables | prefill merges | merges | merge counters (the uploaded image ends
  //      here) | host-buffer page table | partial o | partial lse
  size_t off = kHeaderBytes;
  p.ws.decode_items = off;
  off = align_up(off + p.decode_items.size() * sizeof(WorkItem));
  p.ws.prefill_items = off;
  off = align_up(off + p.prefill_items.size() * sizeof(WorkItem));
  p.ws.prefix_items = off;
  off = align_up(off + p.prefix_items.size() * sizeof(WorkItem));
  p.ws.prefix_tables = off;
  off = align_up(off + p.prefix_tables.size() * sizeof(int32_t));
  p.ws.prefill_merges = off;
  off = align_up(off + p.prefill_merges.size() * sizeof(MergeTask));
  p.ws.merges = off;
  off = align_up(off + p.merges.size() * sizeof(MergeTask));
  // one arrival counter per (merge task, kv head), zero at the start of a
  // run: the CTA that completes a split's last chunk merges it
  p.ws.merge_counters = off;
  off = align_up(off + p.merges.size() * size_t(num_kv_heads) * sizeof(uint32_t));
  p.ws.image_end = off;
  // the page table (plus qo_indptr for a prefill plan) of a host-buffer
  // call, as int32, right after the image: both cross the link in one copy
  p.page_entries = batch > 0 ? page_indptr[batch] : 0;
  const size_t table_ints = size_t(batch + 1) + size_t(p.page_entries) + size_t(batch) +
                            (mode == FI_MODE_PREFILL ? size_t(batch + 1) : 0);
  p.ws.hio_tables = off;
  off = align_up(off + table_ints * sizeof(int32_t));
  p.ws.partial_o = off;
  off = align_up(off + size_t(p.num_slots) * num_qo_heads * head_dim * sizeof(float));
  p.ws.partial_lse = off;
  off = align_up(off + size_t(p.num_slots) * num_qo_heads * sizeof(float));
  p.ws.total = off;
  // host-buffer calls: q and out of the plan's 16-bit dtype, fp32 lse
  const size_t q_bytes = size_t(p.total_q) * num_qo_heads * head_dim * 2;
  p.ws.hio_q = off;
  off = align_up(off + q_bytes);
  p.ws.hio_out = off;
  off = align_up(off + q_bytes);
  p.ws.hio_lse = off;
  off = align_up(off + size_t(p.total_q) * num_qo_heads * sizeof(float));
  p.ws.hio_total = off - p.ws.total;

  *out = std::move(p);
  return FI_OK;
}

}  // namespace fi
