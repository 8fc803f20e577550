// fp64 CPU oracle for block-sparse decode attention over a paged, head-major KV cache.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this code; only the tests, the
// smoke check and the bench's CPU-baseline leg load it.  It shares no code, header, table or
// helper with the CUDA path: it reads the same seeded inputs (bf16 bit patterns, int32
// tables) and computes every step with plain loops in double precision, in the order the
// pages state them, so that a reader can check it against the pages by eye.
//
// Sources (web pages, cited by title and section):
//   [NOSA]  "NOSA: Native and Offloadable Sparse Attention" (technical summary), section
//           "Method 1: the NOSA algorithm" (dual selection, locality guarantee, block-wise
//           implementation, ED-DMA) and "Method 2: the NOSI system" (set-difference).
//   [Spin]  "Unifying Sparse Attention with Hierarchical Memory for Scalable Long-Context LLM
//           Serving", section 2B "Dynamic, locality-aware KV management" (bucketed LRU with
//           64 recency buckets; per-head physical pages).
//   [Lazy]  "LazyAttention" (technical summary), sections "Core idea: deferred positional
//           encoding", "Technical implementation 2. Decoding" and "Mathematical equivalence".
//   [FA]    "How KV sparsity achieves 1.5x acceleration for vLLM" (Novita AI), section
//           "2. Attention modification" (softmax attention, rowmax / l statistics).
//
// Readings of points the pages leave open (each also listed in the design notes):
//   R1 pooling averages keys inside each 16-token sub-block; the max is over the sub-block
//      *scores*; the GQA group's scores are summed before the max.
//   R2 the page holding the newest token (the local page) is always attended, outside the
//      budget, and is never a candidate; candidates are the complete pages before it.
//   R3 eviction scores are per page and ranked directly (pre-exp); exp is never applied.
//   R4 Gamma_e candidates are the pages still alive; unselected candidates die forever;
//      Gamma_q ranks all complete pages outside E (evicted pages allowed).
//   R5 total order for ranking: score descending, then page index ascending.
//   R6 RoPE is the half-split ("rotate-half") form over pairs (x_i, x_{i+64}),
//      theta_i = theta^(-2i/128); stored keys carry only their document-local rotation.
//   R7 packed page word: phys[0:18) | (valid-1)[18:24) | doc slot[24:32).
//   R8 LRU: bucket = min(63, max(0, t - ts) / W); empty slots are bucket 63; hits are
//      touched first; victims are untouched slots in (bucket desc, slot asc) order.
//   R19 prefill step: a prompt row at position n attends to every listed key at a position
//      m <= n; the rows' own keys are listed as a document placed at the first row's position.
//   R20 the prefill's rotated query enters the tensor cores rounded to bf16 (oracle mode 2).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kD = 128;       // head dimension
constexpr int kPage = 64;     // tokens per page (one selection block)
constexpr int kSub = 16;      // tokens per pooling sub-block
constexpr int kNSub = kPage / kSub;
const double kNegInf = -std::numeric_limits<double>::infinity();

// bf16 bit pattern -> exact double (a bf16 is the upper half of an IEEE binary32).
double from_bf16(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

const uint16_t* row_ptr(const uint16_t* plane, int64_t phys, int t) {
  return plane + (phys * kPage + t) * kD;
}

template <class F>
void for_units(int n_units, int nthreads, F f) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  nthreads = std::max(1, std::min(nthreads, n_units));
  std::atomic<int> next{0};
  auto work = [&] {
    for (int i = next.fetch_add(1); i < n_units; i = next.fetch_add(1)) f(i);
  };
  if (nthreads == 1) { work(); return; }
  std::vector<std::thread> th;
  for (int t = 0; t < nthreads; ++t) th.emplace_back(work);
  for (auto& x : th) x.join();
}

// Ranking under R5: true when (a_score, a_page) comes before (b_score, b_page).
bool ranks_before(double as, int ap, double bs, int bp) {
  if (as != bs) return as > bs;
  return ap < bp;
}

// Top-k of `cand` (page ids) under R5 by the score array `sc`, by a plain full sort.
std::vector<int> top_k(const std::vector<int>& cand, const double* sc, int k) {
  std::vector<int> v = cand;
  std::sort(v.begin(), v.end(), [&](int a, int b) { return ranks_before(sc[a], a, sc[b], b); });
  if (static_cast<int>(v.size()) > k) v.resize(k);
  return v;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- packed page word (R7)
// [Lazy] "Technical implementation 2. Decoding": block id and offset are bit-packed into a
// single register-sized word.  Returns 0 on success, -1 if a field is out of range.
int orc_meta_pack(int32_t phys, int32_t valid, int32_t slot, uint32_t* word) {
  if (phys < 0 || phys >= (1 << 18) || valid < 1 || valid > 64 || slot < 0 || slot > 255) return -1;
  *word = static_cast<uint32_t>(phys) | (static_cast<uint32_t>(valid - 1) << 18) |
          (static_cast<uint32_t>(slot) << 24);
  return 0;
}

void orc_meta_unpack(uint32_t word, int32_t* phys, int32_t* valid, int32_t* slot) {
  *phys = static_cast<int32_t>(word & 0x3FFFFu);
  *valid = static_cast<int32_t>((word >> 18) & 0x3Fu) + 1;
  *slot = static_cast<int32_t>(word >> 24);
}

// ---------------------------------------------------------------- A-1 sub-block means
// [NOSA] "Block-wise implementation": first stage of the two-stage pooling, the mean of the
// keys inside each sub-block.  `valid` tokens of the 64-token page hold data; sub-block j
// covers tokens [16j, 16j+16) and averages its cnt[j] valid rows (mean = 0 when cnt[j] = 0).
void orc_page_means(const uint16_t* page, int valid, double* mean, int32_t* cnt) {
  for (int j = 0; j < kNSub; ++j) {
    const int lo = j * kSub, hi = std::min(valid, lo + kSub);
    const int c = std::max(0, hi - lo);
    cnt[j] = c;
    for (int d = 0; d < kD; ++d) {
      double s = 0.0;
      for (int t = lo; t < hi; ++t) s += from_bf16(page[t * kD + d]);
      mean[j * kD + d] = c > 0 ? s / c : 0.0;
    }
  }
}

// Round to the nearest bf16 (8 significant bits), ties to even: the value's binary significand
// m in [1/2, 1) is scaled to [128, 256), rounded to an integer by rint (the default rounding
// mode, nearest-even) and scaled back.  Finite, normal-range inputs.
double orc_round_bf16(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e = 0;
  const double m = std::frexp(x, &e);
  return std::ldexp(std::rint(std::ldexp(m, 8)), e - 8);
}

// ---------------------------------------------------------------- A-2 block scores
// [NOSA] "Block-wise implementation" (two-stage pooling: mean inside sub-blocks, then max to
// the block) with reading R1 for the GQA group:
//   s[p] = max_j  sum_g  (q_g . mean_{p,j}) / sqrt(128)
// for every complete page p before the local page (R2); every other entry is -inf.
// q: G rows of 128 bf16; kplane: the pool plane of this kv head, [n_phys][64][128].
// With summary_bf16 != 0 the stored summary is the sub-block sum rounded to bf16 (cheaper
// scoring at long context, [Spin] 2C): mean = round_bf16(sum) / count.
void orc_score_unit_ex(const uint16_t* q, int G, const uint16_t* kplane, const int32_t* pt_row,
                       int seq_len, int np_out, int summary_bf16, double* s) {
  const int local = (seq_len - 1) / kPage;
  std::vector<double> mean(kNSub * kD);
  int32_t cnt[kNSub];
  const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(kD));
  for (int p = 0; p < np_out; ++p) {
    if (p >= local) { s[p] = kNegInf; continue; }
    orc_page_means(row_ptr(kplane, pt_row[p], 0), kPage, mean.data(), cnt);
    if (summary_bf16)
      for (int j = 0; j < kNSub; ++j)
        for (int d = 0; d < kD; ++d)
          if (cnt[j] > 0) mean[j * kD + d] = orc_round_bf16(mean[j * kD + d] * cnt[j]) / cnt[j];
    double best = kNegInf;
    for (int j = 0; j < kNSub; ++j) {
      double sum_g = 0.0;
      for (int g = 0; g < G; ++g) {
        double dot = 0.0;
        for (int d = 0; d < kD; ++d) dot += from_bf16(q[g * kD + d]) * mean[j * kD + d];
        sum_g += dot;
      }
      best = std::max(best, sum_g * inv_sqrt_d);
    }
    s[p] = best;
  }
}

void orc_score_unit(const uint16_t* q, int G, const uint16_t* kplane, const int32_t* pt_row,
                    int seq_len, int np_out, double* s) {
  orc_score_unit_ex(q, G, kplane, pt_row, seq_len, np_out, 0, s);
}

// ---------------------------------------------------------------- A-3 selection
// [NOSA] "Dual-selection mechanism", "Locality guarantee" and "ED-DMA", with readings R2-R5:
//   candidates C = complete pages 0 .. local-1
//   A = pages of C still alive;  E = top-k_e of A by eviction score (pre-exp, never exp'ed)
//   every page of A outside E dies (alive = 0) and can never enter E again
//   Q = top-k_q of C \ E by query score;  output = sort(E u Q) then the local page.
// alive: one byte per logical page (1 = alive); sel has room for k_e + k_q + 1 entries and
// unused entries are set to -1.
void orc_select_unit(const double* s, const double* e, uint8_t* alive, int np, int seq_len,
                     int k_q, int k_e, int32_t* sel, int32_t* n_sel) {
  const int local = (seq_len - 1) / kPage;
  const int n_cand = std::min(local, np);
  std::vector<int> A, rest;
  for (int p = 0; p < n_cand; ++p)
    if (alive[p]) A.push_back(p);
  std::vector<int> E = top_k(A, e, k_e);
  std::vector<uint8_t> inE(np, 0);
  for (int p : E) inE[p] = 1;
  for (int p : A)
    if (!inE[p]) alive[p] = 0;
  for (int p = 0; p < n_cand; ++p)
    if (!inE[p]) rest.push_back(p);
  std::vector<int> Q = top_k(rest, s, k_q);
  std::vector<int> R = E;
  R.insert(R.end(), Q.begin(), Q.end());
  std::sort(R.begin(), R.end());
  const int stride = k_e + k_q + 1;
  for (int i = 0; i < stride; ++i) sel[i] = -1;
  for (size_t i = 0; i < R.size(); ++i) sel[i] = R[i];
  sel[R.size()] = local;
  *n_sel = static_cast<int32_t>(R.size()) + 1;
}

// ---------------------------------------------------------------- A-4 attention
// [FA] "2. Attention modification": softmax attention written as the plain two-pass form
//   z_t = q . k_t / sqrt(128),  m = max z,  l = sum exp(z_t - m),
//   O = sum exp(z_t - m) v_t / l,  LSE = m + log l   (natural log)
// over every valid token of the listed pages (page i has valid[i] tokens).
// out: G x 128, lse: G.  With no tokens at all, out = 0 and lse = -inf.
void orc_attn_unit(const uint16_t* q, int G, const uint16_t* kplane, const uint16_t* vplane,
                   const int32_t* phys, const int32_t* valid, int n_pages, double* out, double* lse) {
  const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(kD));
  std::vector<double> z;
  for (int g = 0; g < G; ++g) {
    z.clear();
    for (int i = 0; i < n_pages; ++i)
      for (int t = 0; t < valid[i]; ++t) {
        const uint16_t* k = row_ptr(kplane, phys[i], t);
        double dot = 0.0;
        for (int d = 0; d < kD; ++d) dot += from_bf16(q[g * kD + d]) * from_bf16(k[d]);
        z.push_back(dot * inv_sqrt_d);
      }
    if (z.empty()) {
      for (int d = 0; d < kD; ++d) out[g * kD + d] = 0.0;
      lse[g] = kNegInf;
      continue;
    }
    const double m = *std::max_element(z.begin(), z.end());
    double l = 0.0;
    for (double x : z) l += std::exp(x - m);
    for (int d = 0; d < kD; ++d) out[g * kD + d] = 0.0;
    size_t idx = 0;
    for (int i = 0; i < n_pages; ++i)
      for (int t = 0; t < valid[i]; ++t, ++idx) {
        const double w = std::exp(z[idx] - m) / l;
        const uint16_t* v = row_ptr(vplane, phys[i], t);
        for (int d = 0; d < kD; ++d) out[g * kD + d] += w * from_bf16(v[d]);
      }
    lse[g] = m + std::log(l);
  }
}

// ---------------------------------------------------------------- A-5 lazy RoPE
// RoPE rotation by position `pos` (reading R6): for i < 64, with a_i = pos * theta^(-2i/128),
//   y_i = x_i cos a_i - x_{i+64} sin a_i,   y_{i+64} = x_{i+64} cos a_i + x_i sin a_i.
void orc_rope(const double* x, double pos, double theta, double* y) {
  for (int i = 0; i < kD / 2; ++i) {
    const double a = pos * std::pow(theta, -2.0 * i / kD);
    const double c = std::cos(a), s = std::sin(a);
    y[i] = x[i] * c - x[i + kD / 2] * s;
    y[i + kD / 2] = x[i + kD / 2] * c + x[i] * s;
  }
}

// [Lazy] "Mathematical equivalence", materialised side: the query at position qpos is rotated
// by R(qpos); each stored key of document slot i (placed at token offset doc_pos[i]) is copied
// and rotated by R(doc_pos[i]) (it already carries its document-local rotation), then plain
// softmax attention runs on the rotated copies.
void orc_attn_materialised_unit(const uint16_t* q, int G, const uint16_t* kplane,
                                const uint16_t* vplane, const int32_t* phys, const int32_t* valid,
                                const int32_t* slot, int n_pages, int32_t qpos,
                                const int32_t* doc_pos, double theta, double* out, double* lse) {
  const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(kD));
  std::vector<double> keys;  // rotated copies, one row per valid token
  std::vector<int> page_of, tok_of;
  double kin[kD], krot[kD];
  for (int i = 0; i < n_pages; ++i)
    for (int t = 0; t < valid[i]; ++t) {
      const uint16_t* k = row_ptr(kplane, phys[i], t);
      for (int d = 0; d < kD; ++d) kin[d] = from_bf16(k[d]);
      orc_rope(kin, static_cast<double>(doc_pos[slot[i]]), theta, krot);
      keys.insert(keys.end(), krot, krot + kD);
      page_of.push_back(i);
      tok_of.push_back(t);
    }
  const size_t n = page_of.size();
  double qin[kD], qrot[kD];
  std::vector<double> z(n);
  for (int g = 0; g < G; ++g) {
    for (int d = 0; d < kD; ++d) qin[d] = from_bf16(q[g * kD + d]);
    orc_rope(qin, static_cast<double>(qpos), theta, qrot);
    for (int d = 0; d < kD; ++d) out[g * kD + d] = 0.0;
    if (n == 0) { lse[g] = kNegInf; continue; }
    for (size_t r = 0; r < n; ++r) {
      double dot = 0.0;
      for (int d = 0; d < kD; ++d) dot += qrot[d] * keys[r * kD + d];
      z[r] = dot * inv_sqrt_d;
    }
    const double m = *std::max_element(z.begin(), z.end());
    double l = 0.0;
    for (double x : z) l += std::exp(x - m);
    for (size_t r = 0; r < n; ++r) {
      const double w = std::exp(z[r] - m) / l;
      const uint16_t* v = row_ptr(vplane, phys[page_of[r]], tok_of[r]);
      for (int d = 0; d < kD; ++d) out[g * kD + d] += w * from_bf16(v[d]);
    }
    lse[g] = m + std::log(l);
  }
}

// [Lazy] "Technical implementation 2. Decoding", lazy side: keys are used as stored; the query
// is rotated once per document by the relative offset qpos - doc_pos[slot] and that rotated
// query scores every key of the document.
void orc_attn_lazy_unit(const uint16_t* q, int G, const uint16_t* kplane, const uint16_t* vplane,
                        const int32_t* phys, const int32_t* valid, const int32_t* slot, int n_pages,
                        int32_t qpos, const int32_t* doc_pos, double theta, double* out,
                        double* lse) {
  const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(kD));
  double qin[kD], qrot[kD];
  std::vector<double> z;
  for (int g = 0; g < G; ++g) {
    for (int d = 0; d < kD; ++d) qin[d] = from_bf16(q[g * kD + d]);
    z.clear();
    int cur_slot = -1;
    for (int i = 0; i < n_pages; ++i) {
      if (slot[i] != cur_slot) {
        cur_slot = slot[i];
        orc_rope(qin, static_cast<double>(qpos) - doc_pos[cur_slot], theta, qrot);
      }
      for (int t = 0; t < valid[i]; ++t) {
        const uint16_t* k = row_ptr(kplane, phys[i], t);
        double dot = 0.0;
        for (int d = 0; d < kD; ++d) dot += qrot[d] * from_bf16(k[d]);
        z.push_back(dot * inv_sqrt_d);
      }
    }
    for (int d = 0; d < kD; ++d) out[g * kD + d] = 0.0;
    if (z.empty()) { lse[g] = kNegInf; continue; }
    const double m = *std::max_element(z.begin(), z.end());
    double l = 0.0;
    for (double x : z) l += std::exp(x - m);
    size_t idx = 0;
    for (int i = 0; i < n_pages; ++i)
      for (int t = 0; t < valid[i]; ++t, ++idx) {
        const double w = std::exp(z[idx] - m) / l;
        const uint16_t* v = row_ptr(vplane, phys[i], t);
        for (int d = 0; d < kD; ++d) out[g * kD + d] += w * from_bf16(v[d]);
      }
    lse[g] = m + std::log(l);
  }
}

// ---------------------------------------------------------------- A-6 set-difference
// [NOSA] "Method 2: NOSI", optimised memory layout: the blocks to swap in are the selected
// blocks that are not GPU-resident.  missing = sel \ resident (ascending, sel ascending);
// slot[i] = the resident slot holding sel[i], or -1.  resident holds -1 for empty slots.
// missing and slot have `stride` entries; those past the results are set to -1.
void orc_setdiff_unit(const int32_t* resident, int n_slots, const int32_t* sel, int n_sel,
                      int stride, int32_t* missing, int32_t* n_missing, int32_t* slot) {
  for (int i = 0; i < stride; ++i) missing[i] = slot[i] = -1;
  int m = 0;
  for (int i = 0; i < n_sel; ++i) {
    int found = -1;
    for (int s = 0; s < n_slots; ++s)
      if (resident[s] >= 0 && resident[s] == sel[i]) { found = s; break; }
    slot[i] = found;
    if (found < 0) missing[m++] = sel[i];
  }
  *n_missing = m;
}

// ---------------------------------------------------------------- A-7 bucketed LRU
// [Spin] 2B "Bucketed LRU policy": resident pages are grouped into 64 recency buckets by
// their timestamps and evicted a bucket at a time, oldest first (reading R8):
//   1. every hit slot (slot[i] >= 0) is touched: ts = t
//   2. bucket(s) = 63 for an empty slot, else min(63, (t - ts[s]) / W), where a timestamp
//      later than t counts as age 0; hist counts all slots
//   3. victims: the n_missing untouched slots first in (bucket desc, slot asc) order
//   4. missing[i] is installed in victims[i] with ts = t
// victims has `stride` entries; unused entries are -1.
void orc_lru_unit(int32_t* resident, int32_t* ts, int n_slots, const int32_t* slot, int n_sel,
                  const int32_t* missing, int n_missing, int32_t t, int W, int stride,
                  int32_t* victims, int32_t* hist) {
  std::vector<uint8_t> touched(n_slots, 0);
  for (int i = 0; i < n_sel; ++i)
    if (slot[i] >= 0) { ts[slot[i]] = t; touched[slot[i]] = 1; }
  std::vector<int> bucket(n_slots);
  for (int b = 0; b < 64; ++b) hist[b] = 0;
  for (int s = 0; s < n_slots; ++s) {
    if (resident[s] < 0) {
      bucket[s] = 63;
    } else {
      const int64_t age = std::max<int64_t>(0, static_cast<int64_t>(t) - ts[s]);
      bucket[s] = static_cast<int>(std::min<int64_t>(63, age / W));
    }
    hist[bucket[s]] += 1;
  }
  std::vector<int> order;
  for (int s = 0; s < n_slots; ++s)
    if (!touched[s]) order.push_back(s);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return bucket[a] > bucket[b]; });
  for (int i = 0; i < stride; ++i) victims[i] = -1;
  for (int i = 0; i < n_missing && i < static_cast<int>(order.size()); ++i) {
    victims[i] = order[i];
    resident[order[i]] = missing[i];
    ts[order[i]] = t;
  }
}

// ---------------------------------------------------------------- Retrieve (swap-in)
// [NOSA] "Method 2: NOSI": the full KV cache lives in host memory and the selected blocks that
// are not GPU-resident are copied into the buffer slots chosen for them; [Spin] 2A, Retrieve.
// For one unit: for j < n_missing, slot page victims[j] receives host page pt_row[missing[j]]
// (K and V planes of the unit's kv head); then the j-th entry of slot[0 .. n_sel) that is -1
// (the j-th missing page, since the set difference lists them in selection order) becomes
// victims[j].  kslots / vslots point at slot 0 of the unit's own slot range.
void orc_retrieve_unit(const uint16_t* khost, const uint16_t* vhost, const int32_t* pt_row,
                       const int32_t* missing, int n_missing, const int32_t* victims, int32_t* slot,
                       int n_sel, uint16_t* kslots, uint16_t* vslots) {
  const int64_t page_elems = static_cast<int64_t>(kPage) * kD;
  for (int j = 0; j < n_missing; ++j) {
    const int64_t src = static_cast<int64_t>(pt_row[missing[j]]) * page_elems;
    const int64_t dst = static_cast<int64_t>(victims[j]) * page_elems;
    for (int64_t e = 0; e < page_elems; ++e) {
      kslots[dst + e] = khost[src + e];
      vslots[dst + e] = vhost[src + e];
    }
  }
  int j = 0;
  for (int i = 0; i < n_sel; ++i)
    if (slot[i] < 0) slot[i] = victims[j++];
}

// ---------------------------------------------------------------- two-level page directory
// [Spin] 2C "Hierarchical metadata management": the page table of a request is split into
// segments of 2^shift page ids; a directory entry per segment says where that segment lives:
// e >= 0 the device tier (segment e of dev_segs), e <= -2 the host tier (segment -2 - e of
// host_segs), e == -1 nowhere (every page of the range unmapped).  Logical page p of request b is
// entry p mod 2^shift of the segment named by dir[b][p / 2^shift]; -1 when unmapped or when the
// entry names a segment that does not exist.  Writes the flat table [B][np_max].
void orc_dir_to_table(int B, int np_max, const int32_t* dir, int n_dir, int shift, const int32_t* dev_segs,
                      int n_dev, const int32_t* host_segs, int64_t n_host, int32_t* table) {
  const int seg = 1 << shift;
  for (int b = 0; b < B; ++b)
    for (int p = 0; p < np_max; ++p) {
      int32_t v = -1;
      const int s = p / seg;
      if (s < n_dir) {
        const int32_t e = dir[static_cast<int64_t>(b) * n_dir + s];
        if (e >= 0 && e < n_dev) v = dev_segs[static_cast<int64_t>(e) * seg + p % seg];
        if (e <= -2 && -static_cast<int64_t>(e) - 2 < n_host)
          v = host_segs[(-static_cast<int64_t>(e) - 2) * seg + p % seg];
      }
      table[static_cast<int64_t>(b) * np_max + p] = v;
    }
}

// ---------------------------------------------------------------- batch drivers
// The same functions applied to a list of (request, kv head) units, one unit per task on a
// pool of `nthreads` threads (0 = all hardware threads).  Unit u = b * Hk + h.  Pools are
// [Hk][n_phys][64][128]; q is [B][Hq][128]; kv head h serves query heads h*G .. h*G+G-1.

void orc_score_batch_ex(int B, int Hq, int Hk, const uint16_t* q, const uint16_t* kpool, int64_t n_phys,
                        const int32_t* page_table, int np_max, const int32_t* seq_len,
                        const int32_t* units, int n_units, int summary_bf16, double* s, int nthreads) {
  (void)B;
  const int G = Hq / Hk;
  for_units(n_units, nthreads, [&](int i) {
    const int u = units[i], b = u / Hk, h = u % Hk;
    orc_score_unit_ex(q + (static_cast<int64_t>(b) * Hq + h * G) * kD, G,
                      kpool + static_cast<int64_t>(h) * n_phys * kPage * kD,
                      page_table + static_cast<int64_t>(b) * np_max, seq_len[b], np_max, summary_bf16,
                      s + static_cast<int64_t>(u) * np_max);
  });
}

void orc_score_batch(int B, int Hq, int Hk, const uint16_t* q, const uint16_t* kpool, int64_t n_phys,
                     const int32_t* page_table, int np_max, const int32_t* seq_len,
                     const int32_t* units, int n_units, double* s, int nthreads) {
  orc_score_batch_ex(B, Hq, Hk, q, kpool, n_phys, page_table, np_max, seq_len, units, n_units, 0, s, nthreads);
}

void orc_select_batch(int Hk, const double* s, const double* e, uint8_t* alive, int np_max,
                      const int32_t* seq_len, int k_q, int k_e, int32_t* sel, int32_t* n_sel,
                      const int32_t* units, int n_units, int nthreads) {
  const int stride = k_e + k_q + 1;
  for_units(n_units, nthreads, [&](int i) {
    const int u = units[i], b = u / Hk;
    const int64_t o = static_cast<int64_t>(u) * np_max;
    orc_select_unit(s + o, e + o, alive + o, np_max, seq_len[b], k_q, k_e,
                    sel + static_cast<int64_t>(u) * stride, n_sel + u);
  });
}

void orc_sparse_attn_batch(int B, int Hq, int Hk, const uint16_t* q, const uint16_t* kpool,
                           const uint16_t* vpool, int64_t n_phys, const int32_t* page_table,
                           int np_max, const int32_t* sel, const int32_t* n_sel, int sel_stride,
                           const int32_t* seq_len, const int32_t* units, int n_units, double* out,
                           double* lse, int nthreads) {
  (void)B;
  const int G = Hq / Hk;
  for_units(n_units, nthreads, [&](int i) {
    const int u = units[i], b = u / Hk, h = u % Hk;
    const int n = n_sel[u];
    std::vector<int32_t> phys(n), valid(n);
    for (int j = 0; j < n; ++j) {
      const int p = sel[static_cast<int64_t>(u) * sel_stride + j];
      phys[j] = page_table[static_cast<int64_t>(b) * np_max + p];
      valid[j] = std::min(kPage, seq_len[b] - kPage * p);
    }
    const int64_t plane = static_cast<int64_t>(h) * n_phys * kPage * kD;
    const int64_t qo = (static_cast<int64_t>(b) * Hq + h * G);
    orc_attn_unit(q + qo * kD, G, kpool + plane, vpool + plane, phys.data(), valid.data(), n,
                  out + qo * kD, lse + qo);
  });
}

// Lazy-RoPE batch.  phys/valid/slot are [B][meta_heads][np_max] (meta_heads = 1 shares one page
// list across kv heads, or Hk); doc_pos is [B][max_docs].  materialise != 0 runs the
// materialised form, else the lazy form.
void orc_lazy_attn_batch(int B, int Hq, int Hk, const uint16_t* q, const uint16_t* kpool,
                         const uint16_t* vpool, int64_t n_phys, const int32_t* phys,
                         const int32_t* valid, const int32_t* slot, int meta_heads,
                         const int32_t* n_pages, int np_max, const int32_t* qpos,
                         const int32_t* doc_pos, int max_docs, double theta, int materialise,
                         const int32_t* units, int n_units, double* out, double* lse, int nthreads) {
  (void)B;
  const int G = Hq / Hk;
  for_units(n_units, nthreads, [&](int i) {
    const int u = units[i], b = u / Hk, h = u % Hk;
    const int mh = meta_heads == 1 ? 0 : h;
    const int64_t mo = (static_cast<int64_t>(b) * meta_heads + mh) * np_max;
    const int64_t plane = static_cast<int64_t>(h) * n_phys * kPage * kD;
    const int64_t qo = (static_cast<int64_t>(b) * Hq + h * G);
    const int32_t* dp = doc_pos + static_cast<int64_t>(b) * max_docs;
    if (materialise)
      orc_attn_materialised_unit(q + qo * kD, G, kpool + plane, vpool + plane, phys + mo, valid + mo,
                                 slot + mo, n_pages[b], qpos[b], dp, theta, out + qo * kD, lse + qo);
    else
      orc_attn_lazy_unit(q + qo * kD, G, kpool + plane, vpool + plane, phys + mo, valid + mo,
                         slot + mo, n_pages[b], qpos[b], dp, theta, out + qo * kD, lse + qo);
  });
}

// LazyAttention prefill ([Lazy] "Technical implementation 1. Prefilling"): T new query rows
// per request at absolute positions qpos0[b] + t attend over the request's cached document
// pages (no mask: every cached key precedes the rows).  Row t is the single-query attention of
// the functions above at position qpos0[b] + t, so the batch loops over rows.  q is
// [B][T][Hq][128], out [B][T][Hq][128], lse [B][T][Hq]; a work item is (b, t, kv head h),
// numbered ((b * T) + t) * Hk + h.
void orc_lazy_prefill_batch(int B, int T, int Hq, int Hk, const uint16_t* q, const uint16_t* kpool,
                            const uint16_t* vpool, int64_t n_phys, const int32_t* phys,
                            const int32_t* valid, const int32_t* slot, int meta_heads,
                            const int32_t* n_pages, int np_max, const int32_t* qpos0,
                            const int32_t* doc_pos, int max_docs, double theta, int materialise,
                            const int32_t* items, int n_items, double* out, double* lse, int nthreads) {
  (void)B;
  const int G = Hq / Hk;
  for_units(n_items, nthreads, [&](int i) {
    const int it = items[i];
    const int h = it % Hk, bt = it / Hk, t = bt % T, b = bt / T;
    const int mh = meta_heads == 1 ? 0 : h;
    const int64_t mo = (static_cast<int64_t>(b) * meta_heads + mh) * np_max;
    const int64_t plane = static_cast<int64_t>(h) * n_phys * kPage * kD;
    const int64_t qo = static_cast<int64_t>(bt) * Hq + h * G;
    const int32_t* dp = doc_pos + static_cast<int64_t>(b) * max_docs;
    const int32_t pos = qpos0[b] + t;
    if (materialise)
      orc_attn_materialised_unit(q + qo * kD, G, kpool + plane, vpool + plane, phys + mo, valid + mo,
                                 slot + mo, n_pages[b], pos, dp, theta, out + qo * kD, lse + qo);
    else
      orc_attn_lazy_unit(q + qo * kD, G, kpool + plane, vpool + plane, phys + mo, valid + mo,
                         slot + mo, n_pages[b], pos, dp, theta, out + qo * kD, lse + qo);
  });
}

// ---------------------------------------------------------------- the whole RoPE prefill step
// [Lazy] "Technical implementation 1. Prefilling" with reading R19: the prompt's T new rows at
// positions n0 + t attend over every listed key whose absolute position does not come after the
// row, m = doc_pos[slot[i]] + page_start[i] + t <= n.  Cached documents all precede n0, so they are
// seen whole; the rows' own keys, listed as one more document placed at n0 (their document-local
// positions 0 .. T-1), give the causal attention of the rows among themselves in the same softmax.
// mode 0 (materialised, the plain definition): each stored key, which carries its document-local
// rotation, is copied and rotated by R(doc_pos[slot]) to its absolute position, the query by
// R(n), then softmax attention over the visible copies.
// mode 1 (lazy): keys as stored, the query rotated by R(n - doc_pos[slot]) for each document.
// mode 2: mode 1 with the rotated query rounded to bf16 (nearest, ties to even) before the dot
// products -- the precision at which the rotated query enters the tensor cores (reading R20).
void orc_attn_step_unit(const uint16_t* q, int G, const uint16_t* kplane, const uint16_t* vplane,
                        const int32_t* phys, const int32_t* valid, const int32_t* slot, const int32_t* page_start,
                        int n_pages, int32_t qpos, const int32_t* doc_pos, double theta, int mode, double* out,
                        double* lse) {
  const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(kD));
  std::vector<double> z;
  std::vector<const uint16_t*> vrow;
  double qin[kD], qrot[kD], kin[kD], krot[kD];
  for (int g = 0; g < G; ++g) {
    for (int d = 0; d < kD; ++d) qin[d] = from_bf16(q[g * kD + d]);
    if (mode == 0) orc_rope(qin, static_cast<double>(qpos), theta, qrot);
    z.clear();
    vrow.clear();
    int cur_slot = -1;
    for (int i = 0; i < n_pages; ++i) {
      if (mode != 0 && slot[i] != cur_slot) {
        cur_slot = slot[i];
        orc_rope(qin, static_cast<double>(qpos) - doc_pos[cur_slot], theta, qrot);
        if (mode == 2)
          for (int d = 0; d < kD; ++d) qrot[d] = orc_round_bf16(qrot[d]);
      }
      for (int t = 0; t < valid[i]; ++t) {
        const int64_t m = static_cast<int64_t>(doc_pos[slot[i]]) + page_start[i] + t;
        if (m > qpos) continue;   // a key after the row is not attended
        const uint16_t* k = row_ptr(kplane, phys[i], t);
        for (int d = 0; d < kD; ++d) kin[d] = from_bf16(k[d]);
        const double* kk = kin;
        if (mode == 0) {
          orc_rope(kin, static_cast<double>(doc_pos[slot[i]]), theta, krot);
          kk = krot;
        }
        double dot = 0.0;
        for (int d = 0; d < kD; ++d) dot += qrot[d] * kk[d];
        z.push_back(dot * inv_sqrt_d);
        vrow.push_back(row_ptr(vplane, phys[i], t));
      }
    }
    for (int d = 0; d < kD; ++d) out[g * kD + d] = 0.0;
    if (z.empty()) {
      lse[g] = kNegInf;
      continue;
    }
    const double mx = *std::max_element(z.begin(), z.end());
    double l = 0.0;
    for (double x : z) l += std::exp(x - mx);
    for (size_t r = 0; r < z.size(); ++r) {
      const double w = std::exp(z[r] - mx) / l;
      for (int d = 0; d < kD; ++d) out[g * kD + d] += w * from_bf16(vrow[r][d]);
    }
    lse[g] = mx + std::log(l);
  }
}

// The step for every (request, row, kv head) work item listed, numbered ((b * T) + t) * Hk + h;
// arrays as in orc_lazy_prefill_batch plus page_start ([B][meta_heads][np_max], the document-local
// position of each listed page's first token).
void orc_prefill_step_batch(int B, int T, int Hq, int Hk, const uint16_t* q, const uint16_t* kpool,
                            const uint16_t* vpool, int64_t n_phys, const int32_t* phys, const int32_t* valid,
                            const int32_t* slot, const int32_t* page_start, int meta_heads, const int32_t* n_pages,
                            int np_max, const int32_t* qpos0, const int32_t* doc_pos, int max_docs, double theta,
                            int mode, const int32_t* items, int n_items, double* out, double* lse, int nthreads) {
  (void)B;
  const int G = Hq / Hk;
  for_units(n_items, nthreads, [&](int i) {
    const int it = items[i];
    const int h = it % Hk, bt = it / Hk, t = bt % T, b = bt / T;
    const int mh = meta_heads == 1 ? 0 : h;
    const int64_t mo = (static_cast<int64_t>(b) * meta_heads + mh) * np_max;
    const int64_t plane = static_cast<int64_t>(h) * n_phys * kPage * kD;
    const int64_t qo = static_cast<int64_t>(bt) * Hq + h * G;
    orc_attn_step_unit(q + qo * kD, G, kpool + plane, vpool + plane, phys + mo, valid + mo, slot + mo,
                       page_start + mo, n_pages[b], qpos0[b] + t, doc_pos + static_cast<int64_t>(b) * max_docs,
                       theta, mode, out + qo * kD, lse + qo);
  });
}

// ---------------------------------------------------------------- ALiBi prefill
// [Lazy] "Key contributions" 4 (the mechanism carries over to other relative position encodings,
// ALiBi among them), reading R18: keys are stored with no positional transform; the key at
// document-local position page_start[i] + t of document slot[i], placed at token offset
// doc_pos[slot[i]], sits at m = doc_pos[slot[i]] + page_start[i] + t; the query row at position
// n scores it as q . k / sqrt(128) - slope * (n - m) (the linear bias of ALiBi, one slope per
// query head, natural-log units), and plain softmax attention follows over the keys that do not
// come after the row (m <= n; reading R19): cached documents all precede the rows, and the rows'
// own keys listed as a document at offset n0 give the causal part of the prefill step.
// q: G query heads of 128 bf16; slopes: their G slopes.
void orc_alibi_attn_unit(const uint16_t* q, int G, const float* slopes, const uint16_t* kplane,
                         const uint16_t* vplane, const int32_t* phys, const int32_t* valid, const int32_t* slot,
                         const int32_t* page_start, int n_pages, int32_t qpos, const int32_t* doc_pos,
                         double* out, double* lse) {
  const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(kD));
  std::vector<double> z;
  std::vector<const uint16_t*> vrow;
  for (int g = 0; g < G; ++g) {
    const double slope = slopes[g];
    z.clear();
    vrow.clear();
    for (int i = 0; i < n_pages; ++i)
      for (int t = 0; t < valid[i]; ++t) {
        const double m = static_cast<double>(doc_pos[slot[i]]) + page_start[i] + t;
        if (m > qpos) continue;   // a key after the row is not attended
        const uint16_t* k = row_ptr(kplane, phys[i], t);
        double dot = 0.0;
        for (int d = 0; d < kD; ++d) dot += from_bf16(q[g * kD + d]) * from_bf16(k[d]);
        z.push_back(dot * inv_sqrt_d - slope * (static_cast<double>(qpos) - m));
        vrow.push_back(row_ptr(vplane, phys[i], t));
      }
    for (int d = 0; d < kD; ++d) out[g * kD + d] = 0.0;
    if (z.empty()) {
      lse[g] = kNegInf;
      continue;
    }
    const double mx = *std::max_element(z.begin(), z.end());
    double l = 0.0;
    for (double x : z) l += std::exp(x - mx);
    for (size_t r = 0; r < z.size(); ++r) {
      const double w = std::exp(z[r] - mx) / l;
      for (int d = 0; d < kD; ++d) out[g * kD + d] += w * from_bf16(vrow[r][d]);
    }
    lse[g] = mx + std::log(l);
  }
}

// ALiBi prefill batch: the prefill of orc_lazy_prefill_batch with the bias above instead of the
// rotation; page_start is [B][meta_heads][np_max] like phys, slopes is [Hq].
void orc_alibi_prefill_batch(int B, int T, int Hq, int Hk, const uint16_t* q, const uint16_t* kpool,
                             const uint16_t* vpool, int64_t n_phys, const int32_t* phys, const int32_t* valid,
                             const int32_t* slot, const int32_t* page_start, int meta_heads,
                             const int32_t* n_pages, int np_max, const int32_t* qpos0, const int32_t* doc_pos,
                             int max_docs, const float* slopes, const int32_t* items, int n_items, double* out,
                             double* lse, int nthreads) {
  (void)B;
  const int G = Hq / Hk;
  for_units(n_items, nthreads, [&](int i) {
    const int it = items[i];
    const int h = it % Hk, bt = it / Hk, t = bt % T, b = bt / T;
    const int mh = meta_heads == 1 ? 0 : h;
    const int64_t mo = (static_cast<int64_t>(b) * meta_heads + mh) * np_max;
    const int64_t plane = static_cast<int64_t>(h) * n_phys * kPage * kD;
    const int64_t qo = static_cast<int64_t>(bt) * Hq + h * G;
    orc_alibi_attn_unit(q + qo * kD, G, slopes + h * G, kpool + plane, vpool + plane, phys + mo, valid + mo,
                        slot + mo, page_start + mo, n_pages[b], qpos0[b] + t,
                        doc_pos + static_cast<int64_t>(b) * max_docs, out + qo * kD, lse + qo);
  });
}

// ---------------------------------------------------------------- column score S
// [FA] "2. Attention modification" (the PyramidKV-style sparsification score, reading R16): the
// last alpha rows of a prompt of n tokens, at positions n - alpha + j, attend causally over the
// prompt's keys; with A[j][i] = softmax over i <= n - alpha + j of q_j . k_i / sqrt(128),
//   S[i] = sum_j A[j][i]          (i < n; a key after a row's position gets nothing from it).
// Computed the two-pass way the page describes: each row's log-sum-exp first (rowmax and l),
// then every probability from it.  q: alpha rows of 128 bf16 (one query head); kplane: the pool
// plane of its kv head; pt_row: the request's page table; S: n_out entries (>= n are 0).
void orc_column_scores_unit(const uint16_t* q, int q_stride, int alpha, const uint16_t* kplane,
                            const int32_t* pt_row, int n, int n_out, double* S) {
  const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(kD));
  for (int i = 0; i < n_out; ++i) S[i] = 0.0;
  std::vector<double> z(n);
  for (int j = 0; j < alpha; ++j) {
    const int pos = n - alpha + j;
    if (pos < 0) continue;
    const uint16_t* qj = q + static_cast<int64_t>(j) * q_stride;
    for (int i = 0; i <= pos; ++i) {
      const uint16_t* k = row_ptr(kplane, pt_row[i / kPage], i % kPage);
      double dot = 0.0;
      for (int d = 0; d < kD; ++d) dot += from_bf16(qj[d]) * from_bf16(k[d]);
      z[i] = dot * inv_sqrt_d;
    }
    double m = kNegInf;
    for (int i = 0; i <= pos; ++i) m = std::max(m, z[i]);
    double l = 0.0;
    for (int i = 0; i <= pos; ++i) l += std::exp(z[i] - m);
    const double lse = m + std::log(l);
    for (int i = 0; i <= pos; ++i) S[i] += std::exp(z[i] - lse);
  }
}

// Column scores for every (request, query head) listed: q is [B][alpha][Hq][128], S is
// [B][Hq][n_out]; request b's prompt has seq_len[b] tokens in pages page_table[b][...].
void orc_column_scores_batch(int B, int Hq, int Hk, int alpha, const uint16_t* q, const uint16_t* kpool,
                             int64_t n_phys, const int32_t* page_table, int np_max, const int32_t* seq_len,
                             int n_out, const int32_t* items, int n_items, double* S, int nthreads) {
  (void)B;
  const int G = Hq / Hk;
  for_units(n_items, nthreads, [&](int i) {
    const int it = items[i], b = it / Hq, hq = it % Hq, h = hq / G;
    orc_column_scores_unit(q + (static_cast<int64_t>(b) * alpha * Hq + hq) * kD, Hq * kD, alpha,
                           kpool + static_cast<int64_t>(h) * n_phys * kPage * kD,
                           page_table + static_cast<int64_t>(b) * np_max, seq_len[b], n_out,
                           S + static_cast<int64_t>(it) * n_out);
  });
}

// The same score with each row's log-sum-exp given instead of computed ([FA] "2. Attention
// modification": the FlashAttention pass already produced rowmax and l, so the score needs only
// the probability pass).  With lse_j the natural-log LSE the caller supplies for row j,
//   S[i] = sum over rows j with i <= n - alpha + j of exp(q_j . k_i / sqrt(128) - lse_j).
// When lse_j is the row's own log-sum-exp this is orc_column_scores_unit exactly.
void orc_column_scores_given_lse_unit(const uint16_t* q, int q_stride, int alpha, const double* lse,
                                      int lse_stride, const uint16_t* kplane, const int32_t* pt_row, int n,
                                      int n_out, double* S) {
  const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(kD));
  for (int i = 0; i < n_out; ++i) S[i] = 0.0;
  for (int j = 0; j < alpha; ++j) {
    const int pos = n - alpha + j;
    if (pos < 0) continue;
    const uint16_t* qj = q + static_cast<int64_t>(j) * q_stride;
    const double lj = lse[static_cast<int64_t>(j) * lse_stride];
    for (int i = 0; i <= pos; ++i) {
      const uint16_t* k = row_ptr(kplane, pt_row[i / kPage], i % kPage);
      double dot = 0.0;
      for (int d = 0; d < kD; ++d) dot += from_bf16(qj[d]) * from_bf16(k[d]);
      S[i] += std::exp(dot * inv_sqrt_d - lj);
    }
  }
}

// Batch driver of the given-LSE form: lse is [B][alpha][Hq] (natural log), the rest as above.
void orc_column_scores_given_lse_batch(int B, int Hq, int Hk, int alpha, const uint16_t* q, const double* lse,
                                       const uint16_t* kpool, int64_t n_phys, const int32_t* page_table,
                                       int np_max, const int32_t* seq_len, int n_out, const int32_t* items,
                                       int n_items, double* S, int nthreads) {
  (void)B;
  const int G = Hq / Hk;
  for_units(n_items, nthreads, [&](int i) {
    const int it = items[i], b = it / Hq, hq = it % Hq, h = hq / G;
    orc_column_scores_given_lse_unit(q + (static_cast<int64_t>(b) * alpha * Hq + hq) * kD, Hq * kD, alpha,
                                     lse + static_cast<int64_t>(b) * alpha * Hq + hq, Hq,
                                     kpool + static_cast<int64_t>(h) * n_phys * kPage * kD,
                                     page_table + static_cast<int64_t>(b) * np_max, seq_len[b], n_out,
                                     S + static_cast<int64_t>(it) * n_out);
  });
}

// Retrieve for every unit.  Host pools [Hk][n_host][64][128]; slot pools [Hk][n_slot_pages][64][128]
// with unit (b, h)'s slots at pages b * n_slots .. b * n_slots + n_slots - 1 of plane h.
void orc_retrieve_batch(int B, int Hk, const uint16_t* khost, const uint16_t* vhost, int64_t n_host,
                        const int32_t* page_table, int np_max, const int32_t* missing,
                        const int32_t* n_missing, const int32_t* victims, int32_t* slot,
                        const int32_t* n_sel, int sel_stride, uint16_t* kslots, uint16_t* vslots,
                        int64_t n_slot_pages, int n_slots, int nthreads) {
  const int64_t page_elems = static_cast<int64_t>(kPage) * kD;
  for_units(B * Hk, nthreads, [&](int u) {
    const int b = u / Hk, h = u % Hk;
    const int64_t so = static_cast<int64_t>(u) * sel_stride;
    const int64_t hplane = static_cast<int64_t>(h) * n_host * page_elems;
    const int64_t splane = (static_cast<int64_t>(h) * n_slot_pages + static_cast<int64_t>(b) * n_slots) *
                           page_elems;
    orc_retrieve_unit(khost + hplane, vhost + hplane, page_table + static_cast<int64_t>(b) * np_max,
                      missing + so, n_missing[u], victims + so, slot + so, n_sel[u], kslots + splane,
                      vslots + splane);
  });
}

// Sparse attention reading the selected pages from their slots: page sel[u][j] of unit (b, h)
// is slot page b * n_slots + slot[u][j] of plane h; its valid tokens follow from seq_len.
void orc_slot_attn_batch(int B, int Hq, int Hk, const uint16_t* q, const uint16_t* kslots,
                         const uint16_t* vslots, int64_t n_slot_pages, const int32_t* sel,
                         const int32_t* slot, const int32_t* n_sel, int sel_stride, int n_slots,
                         const int32_t* seq_len, const int32_t* units, int n_units, double* out,
                         double* lse, int nthreads) {
  (void)B;
  const int G = Hq / Hk;
  for_units(n_units, nthreads, [&](int i) {
    const int u = units[i], b = u / Hk, h = u % Hk;
    const int n = n_sel[u];
    std::vector<int32_t> phys(n), valid(n);
    for (int j = 0; j < n; ++j) {
      const int64_t e = static_cast<int64_t>(u) * sel_stride + j;
      phys[j] = b * n_slots + slot[e];
      valid[j] = std::min(kPage, seq_len[b] - kPage * sel[e]);
    }
    const int64_t plane = static_cast<int64_t>(h) * n_slot_pages * kPage * kD;
    const int64_t qo = (static_cast<int64_t>(b) * Hq + h * G);
    orc_attn_unit(q + qo * kD, G, kslots + plane, vslots + plane, phys.data(), valid.data(), n,
                  out + qo * kD, lse + qo);
  });
}

void orc_setdiff_batch(const int32_t* resident, int n_slots, const int32_t* sel, const int32_t* n_sel,
                       int sel_stride, int n_units, int32_t* missing, int32_t* n_missing,
                       int32_t* slot, int nthreads) {
  for_units(n_units, nthreads, [&](int u) {
    const int64_t so = static_cast<int64_t>(u) * sel_stride;
    orc_setdiff_unit(resident + static_cast<int64_t>(u) * n_slots, n_slots, sel + so, n_sel[u],
                     sel_stride, missing + so, n_missing + u, slot + so);
  });
}

void orc_lru_batch(int32_t* resident, int32_t* ts, int n_slots, const int32_t* slot,
                   const int32_t* n_sel, const int32_t* missing, const int32_t* n_missing,
                   int sel_stride, int n_units, int32_t t, int W, int32_t* victims, int32_t* hist,
                   int nthreads) {
  for_units(n_units, nthreads, [&](int u) {
    const int64_t so = static_cast<int64_t>(u) * sel_stride;
    const int64_t ro = static_cast<int64_t>(u) * n_slots;
    orc_lru_unit(resident + ro, ts + ro, n_slots, slot + so, n_sel[u], missing + so, n_missing[u], t,
                 W, sel_stride, victims + so, hist + static_cast<int64_t>(u) * 64);
  });
}

}  // extern "C"
