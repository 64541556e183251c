// Host plan compiler: validates a naming and lowers it to the work tables of the two
// datapaths (zero-copy tiles; staged units, items and warps).
//
// Source: Purlin article, "The Purlin PDF describes a three-layer design" — SNAC derives
// the coordination (who waits for whom) from the collective's naming. Here that means:
// every consumed name is cut into pieces; producers of a name stage and notify per piece,
// its consumers wait for (or validate) exactly those producers' flags.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <unordered_map>
#include <vector>

#include "coll_internal.h"

namespace {

int esize_of(int dt) {
  switch (dt) {
    case COLL_BF16: return 2;
    case COLL_F32: return 4;
    case COLL_BYTES: return 1;
    default: return 0;
  }
}

struct NameInfo {
  uint64_t count = 0;
  std::vector<uint32_t> prod;  // indices into in_segs
  std::vector<uint32_t> cons;  // indices into out_segs
};

}  // namespace

extern "C" int coll_config_default(coll_config_t *cfg) {
  if (!cfg) return COLL_EINVAL;
  memset(cfg, 0, sizeof(*cfg));
  cfg->protocol = COLL_PROTO_SPEC;
  cfg->datapath = COLL_DP_ONESHOT;
  cfg->zero_copy = 0;
  cfg->spec_check = COLL_SPEC_TAGGED_RELAXED;
  cfg->spec_delay_ns = -1;
  cfg->unit_bytes = 0;
  cfg->inject_rank = -1;
  return COLL_OK;
}

static int check_config(const coll_config_t &c) {
  if (c.protocol < 0 || c.protocol > 3) return COLL_EINVAL;
  if (c.datapath < 0 || c.datapath > 2) return COLL_EINVAL;
  // the pull needs the staged exchange buffers; tagged data has no flags to pull on
  if (c.datapath == COLL_DP_TWOSHOT_PULL && (c.zero_copy || c.protocol == COLL_PROTO_LL))
    return COLL_EINVAL;
  if (c.zero_copy < 0 || c.zero_copy > 1) return COLL_EINVAL;
  if (c.spec_check < 0 || c.spec_check > 2) return COLL_EINVAL;
  if (c.unit_bytes != 0 && (c.unit_bytes < 64 || c.unit_bytes > 512 || (c.unit_bytes & 15)))
    return COLL_EINVAL;
  if (c.warps_per_rank < 0 || c.ctas < 0) return COLL_EINVAL;
  if (c.tile_bytes < 0 || (c.tile_bytes % 16) != 0) return COLL_EINVAL;
  if (c.inject_prob_ppm > 1000000u) return COLL_EINVAL;
  if (c.chain < 0 || c.chain > 1 || c.reserved3 != 0) return COLL_EINVAL;
  if (c.spec_delay_ns < -1 || c.spec_delay_ns > 100000) return COLL_EINVAL;
  if (c.reduce_order < 0 || c.reduce_order > 1) return COLL_EINVAL;
  // the staged engine always sums in rank order
  if (c.reduce_order != COLL_ORDER_RANK && !c.zero_copy) return COLL_EINVAL;
  return COLL_OK;
}

int coll_compile(int R, int op, int dtype, const coll_seg_t *in_segs, size_t n_in,
                 const uint64_t *in_len, const coll_seg_t *out_segs, size_t n_out,
                 const uint64_t *out_len, const coll_config_t *cfg_in, int max_warps,
                 int num_sms, coll_compiled *out) {
  coll_compiled c;
  if (cfg_in) c.cfg = *cfg_in; else coll_config_default(&c.cfg);
  const coll_config_t &cfg = c.cfg;

  // 1. arguments
  if (R < 1 || R > COLL_MAX_RANKS) return COLL_EINVAL;
  if (op != COLL_OP_COPY && op != COLL_OP_SUM) return COLL_EINVAL;
  const int es = esize_of(dtype);
  if (es == 0) return COLL_EINVAL;
  if (op == COLL_OP_SUM && dtype == COLL_BYTES) return COLL_EINVAL;
  if (!in_len || !out_len) return COLL_EINVAL;
  if ((n_in && !in_segs) || (n_out && !out_segs)) return COLL_EINVAL;
  if (n_in > 0xFFFFFFF0u || n_out > 0xFFFFFFF0u) return COLL_EINVAL;
  // byte sizes (elements x element size, times ranks) must stay far from 64-bit overflow
  for (int r = 0; r < R; ++r)
    if (in_len[r] > COLL_MAX_ELEMS || out_len[r] > COLL_MAX_ELEMS) return COLL_EBOUNDS;
  // 2. segments: rank, count, reserved
  for (size_t i = 0; i < n_in + n_out; ++i) {
    const coll_seg_t &s = i < n_in ? in_segs[i] : out_segs[i - n_in];
    if (s.rank < 0 || s.rank >= R || s.count == 0 || s.reserved != 0) return COLL_EINVAL;
  }
  // 3. bounds
  for (size_t i = 0; i < n_in; ++i) {
    const coll_seg_t &s = in_segs[i];
    const uint64_t L = in_len[s.rank];
    if (s.offset > L || s.count > L - s.offset) return COLL_EBOUNDS;
  }
  for (size_t i = 0; i < n_out; ++i) {
    const coll_seg_t &s = out_segs[i];
    const uint64_t L = out_len[s.rank];
    if (s.offset > L || s.count > L - s.offset) return COLL_EBOUNDS;
  }
  // 4. one count per name
  std::unordered_map<uint64_t, uint64_t> count_of;
  count_of.reserve(n_in + n_out);
  for (size_t i = 0; i < n_in + n_out; ++i) {
    const coll_seg_t &s = i < n_in ? in_segs[i] : out_segs[i - n_in];
    auto it = count_of.emplace(s.name, s.count);
    if (it.first->second != s.count) return COLL_ELEN;
  }
  // 5. producers per consumed name
  std::unordered_map<uint64_t, uint32_t> name_idx;  // consumed names, first-appearance order
  std::vector<NameInfo> names;
  for (size_t i = 0; i < n_out; ++i) {
    auto it = name_idx.emplace(out_segs[i].name, (uint32_t)names.size());
    if (it.second) {
      names.emplace_back();
      names.back().count = out_segs[i].count;
    }
    names[it.first->second].cons.push_back((uint32_t)i);
  }
  for (size_t i = 0; i < n_in; ++i) {
    auto it = name_idx.find(in_segs[i].name);
    if (it != name_idx.end()) names[it->second].prod.push_back((uint32_t)i);
  }
  for (auto &nm : names) {
    if (nm.prod.empty() || (op == COLL_OP_COPY && nm.prod.size() != 1)) return COLL_ENAME;
  }
  // 6. outputs of one rank must not overlap
  {
    std::vector<std::vector<std::pair<uint64_t, uint64_t>>> per(R);
    for (size_t i = 0; i < n_out; ++i)
      per[out_segs[i].rank].emplace_back(out_segs[i].offset, out_segs[i].count);
    for (auto &v : per) {
      std::sort(v.begin(), v.end());
      for (size_t k = 1; k < v.size(); ++k)
        if (v[k - 1].first + v[k - 1].second > v[k].first) return COLL_EOVERLAP;
    }
  }
  // config
  if (int e = check_config(cfg)) return e;
  // fan-in / fan-out limits of the device tables
  for (auto &nm : names)
    if (nm.prod.size() > COLL_MAX_FANIN || nm.cons.size() > COLL_MAX_FANOUT) return COLL_EINVAL;
  // staged plans move 16-byte vectors between exchange slots
  const bool staged = cfg.zero_copy == 0;
  if (staged) {
    for (size_t i = 0; i < n_in + n_out; ++i) {
      const coll_seg_t &s = i < n_in ? in_segs[i] : out_segs[i - n_in];
      if (((s.offset * es) & 15u) || ((s.count * es) & 15u)) return COLL_EALIGN;
    }
  }

  // ---------------- common bookkeeping
  c.R = R;
  c.op = op;
  c.dtype = dtype;
  c.esize = es;
  c.in_bytes.resize(R);
  c.out_bytes.resize(R);
  c.in_used.assign(R, 0);
  c.out_used.assign(R, 0);
  for (int r = 0; r < R; ++r) {
    c.in_bytes[r] = in_len[r] * es;
    c.out_bytes[r] = out_len[r] * es;
  }
  const bool sum = op == COLL_OP_SUM;
  const bool pull = sum && cfg.datapath == COLL_DP_TWOSHOT_PULL;
  const bool twoshot = sum && (cfg.datapath == COLL_DP_TWOSHOT || pull);
  c.n_names = names.size();
  for (auto &nm : names) {
    // producers in (rank, offset) order: the fixed summation order
    std::stable_sort(nm.prod.begin(), nm.prod.end(), [&](uint32_t a, uint32_t b) {
      if (in_segs[a].rank != in_segs[b].rank) return in_segs[a].rank < in_segs[b].rank;
      return in_segs[a].offset < in_segs[b].offset;
    });
    const uint64_t bytes = nm.count * es;
    c.min_bytes += bytes * (nm.prod.size() + nm.cons.size());
    for (uint32_t p : nm.prod) c.in_used[in_segs[p].rank] = 1;
    for (uint32_t q : nm.cons) c.out_used[out_segs[q].rank] = 1;
  }

  auto ref_of = [&](const coll_seg_t &s) {
    coll_ref_t r;
    r.rank = (uint32_t)s.rank;
    r.pad = 0;
    r.off = s.offset * es;
    return r;
  };

  if (!staged) {
    // ---------------- zero-copy: jobs and tiles
    // One warp per tile. Default tile: the largest power of two (512 B .. 32 KiB) that
    // still gives about four tiles per resident warp (32 per SM), so small collectives
    // spread over every SM and large ones keep per-tile overhead low.
    uint64_t job_bytes = 0, src_bytes = 0;
    uint32_t maxsrc = 0, maxdst = 0;
    bool aligned = true;
    for (auto &nm : names) {
      const uint64_t njobs = (!sum || twoshot) ? 1u : nm.cons.size();
      if (njobs > 1) c.zc_keep = true;
      job_bytes += nm.count * es * njobs;
      src_bytes += nm.count * es * njobs * (sum ? nm.prod.size() : 1u);
      maxsrc = std::max<uint32_t>(maxsrc, sum ? (uint32_t)nm.prod.size() : 1u);
      maxdst = std::max<uint32_t>(maxdst, (!sum || twoshot) ? (uint32_t)nm.cons.size() : 1u);
      if ((nm.count * es) & 15u) aligned = false;
    }
    for (size_t i = 0; i < n_in + n_out && aligned; ++i) {
      const coll_seg_t &sg = i < n_in ? in_segs[i] : out_segs[i - n_in];
      if ((sg.offset * es) & 15u) aligned = false;
    }
    const uint64_t sms = (uint64_t)(num_sms > 0 ? num_sms : 152);
    // Large aligned plans use the bulk (TMA) ring: one CTA per SM, tiles of
    // 32 KiB / (producers rounded up to a power of two), at least four tiles per CTA.
    // Jobs that write each loaded byte to four or more destinations (broadcast,
    // all-gather, MoE dispatch) take longest per tile; their tiles are capped at 16 KiB,
    // which doubles the tiles per CTA for the same bytes in flight (measured: broadcast
    // 64 MiB 0.85 -> 0.91, all-gather 16 MiB 0.89 -> 0.93). Plans whose inputs are re-read
    // (one-shot sums) take most of their bytes from L2, where larger copies move faster:
    // their stages hold 64 KiB (one-shot all-reduce 8 x 32 MiB 0.29 -> 0.34; the plans
    // that stream from DRAM keep six stages of 32 KiB, which measured better for them).
    // The ring's stages are sized for the largest producer count; jobs with fewer
    // producers leave stage space idle, so the ring is used only when jobs fill at least
    // three quarters of it on average (uniform collectives); uneven ones (MoE combine)
    // stay on the warp kernel.
    const uint64_t bulk_min = cfg.tma_min_bytes ? cfg.tma_min_bytes : (4ull << 20);
    const bool filled = maxsrc > 0 && src_bytes * 4 >= job_bytes * maxsrc * 3;
    c.bulk = aligned && maxsrc >= 1 && maxsrc <= COLL_BULK_MAX_SRC &&
             maxdst <= COLL_BULK_MAX_DST && job_bytes >= bulk_min && !cfg.tile_bytes &&
             (filled || cfg.tma_min_bytes != 0);
    uint64_t T = cfg.tile_bytes ? (uint64_t)cfg.tile_bytes : 0;
    if (c.bulk) {
      uint32_t p2 = 1;
      while (p2 < maxsrc) p2 *= 2;
      const uint64_t stage_cap = c.zc_keep ? 65536u : 32768u;
      const uint64_t cap = maxdst >= 4u * maxsrc ? std::min<uint64_t>(16384u, stage_cap / p2)
                                                 : stage_cap / p2;
      const uint64_t want = job_bytes / (4u * sms);
      T = 1024;
      while (T < cap && T * 2 <= want) T *= 2;
      c.bulk_slot = (uint32_t)T;
      c.bulk_maxsrc = maxsrc;
      // as many stages as fit in 192 KiB of shared memory (2..12)
      const uint64_t stage = (uint64_t)maxsrc * T;
      c.bulk_stages = (uint32_t)std::max<uint64_t>(2, std::min<uint64_t>(12, (192u << 10) / stage));
      // Jobs with at least as many consumers as producers finish faster when the ring
      // claims its last tiles two at a time. Many-to-one sums that read each input once
      // (reduce-scatter, reduce to root) lose with such small claims and gain, in long
      // runs, with guided ones; the one-shot all-reduce, whose inputs are re-read, deals
      // every tile round-robin (all measured).
      c.bulk_tail = maxdst >= maxsrc ? 1u : (c.zc_keep ? 0u : 2u);
    } else if (!T) {
      // One warp per tile: the largest power of two (512 B .. 32 KiB) that still gives
      // about four tiles per resident warp (32 per SM).
      const uint64_t want = job_bytes / (4u * sms * 32u);
      T = 512;
      while (T < 32768u && T * 2 <= want) T *= 2;
    }
    // On the ring, a plan whose jobs write each piece to eight or more destinations and that
    // would give a CTA fewer than 16 tiles splits each such job into two, each writing to half
    // of the destinations (the second reads the piece again, from L2). A 16 MiB broadcast
    // (7 tiles per CTA, each writing 128 KiB) then balances its SMs better: 0.68-0.72 /
    // 0.78 -> 0.78 / 0.85 single / back to back, measured; with 27 or more tiles per CTA
    // the split did not pay.
    const bool dsplit = c.bulk && T && job_bytes / T < 16u * sms;
    for (auto &nm : names) {
      const uint64_t bytes = nm.count * es;
      const uint32_t job0 = (uint32_t)c.jobs.size();
      const uint32_t src0 = (uint32_t)c.refs.size();
      const uint32_t nsrc = sum ? (uint32_t)nm.prod.size() : 1u;
      for (uint32_t k = 0; k < nsrc; ++k) c.refs.push_back(ref_of(in_segs[nm.prod[k]]));
      if (!sum || twoshot) {
        const uint32_t nd = (uint32_t)nm.cons.size();
        const uint32_t G = dsplit && nd >= 8u && nd >= 8u * nsrc ? 2u : 1u;
        for (uint32_t g = 0; g < G; ++g) {
          const uint32_t d0 = nd * g / G, d1 = nd * (g + 1) / G;
          coll_job_t j;
          j.src0 = src0;
          j.nsrc = nsrc;
          j.dst0 = (uint32_t)c.refs.size();
          j.ndst = d1 - d0;
          for (uint32_t q = d0; q < d1; ++q) c.refs.push_back(ref_of(out_segs[nm.cons[q]]));
          c.jobs.push_back(j);
        }
      } else {
        for (uint32_t q : nm.cons) {
          coll_job_t j;
          j.src0 = src0;
          j.nsrc = nsrc;
          j.dst0 = (uint32_t)c.refs.size();
          j.ndst = 1;
          c.refs.push_back(ref_of(out_segs[q]));
          c.jobs.push_back(j);
        }
      }
      const uint32_t job1 = (uint32_t)c.jobs.size();
      // chunk-major, job-minor: consumers of one chunk run close together in time, so
      // a oneshot's repeated reads of the same sources hit L2
      for (uint64_t start = 0; start < bytes; start += T) {
        const uint64_t nb = std::min<uint64_t>(T, bytes - start);
        for (uint32_t j = job0; j < job1; ++j) {
          coll_tile_t t;
          t.job = j;
          t.nbytes = (uint32_t)nb;
          t.start = start;
          c.tiles.push_back(t);
        }
      }
    }
    if (c.tiles.size() > 0xFFFFFFF0ull) return COLL_EINVAL;
    // inline tile records whenever every job fits them (the bulk ring needs them; the warp
    // kernel uses them when present)
    if (maxsrc <= COLL_BULK_MAX_SRC && maxdst <= COLL_BULK_MAX_DST) {
      c.btiles.resize(c.tiles.size());
      for (size_t i = 0; i < c.tiles.size(); ++i) {
        const coll_tile_t &t = c.tiles[i];
        const coll_job_t &j = c.jobs[t.job];
        coll_btile_t &b = c.btiles[i];
        memset(&b, 0, sizeof(b));
        b.start = t.start;
        b.nbytes = t.nbytes;
        b.nsrc = (uint16_t)j.nsrc;
        b.ndst = (uint16_t)j.ndst;
        for (uint32_t k = 0; k < j.nsrc; ++k)
          b.ref[k] = COLL_BULK_REF(c.refs[j.src0 + k].rank, c.refs[j.src0 + k].off);
        for (uint32_t k = 0; k < j.ndst; ++k)
          b.ref[COLL_BULK_MAX_SRC + k] =
              COLL_BULK_REF(c.refs[j.dst0 + k].rank, c.refs[j.dst0 + k].off);
      }
    }
    *out = std::move(c);
    return COLL_OK;
  }

  // ---------------- staged: units, items, warps
  const uint32_t U = cfg.unit_bytes ? (uint32_t)cfg.unit_bytes : 512u;
  std::vector<std::vector<coll_item_t>> S(R), C(R), P(R);  // per-rank stage / consume / pull
  std::vector<uint32_t> unit_owner;
  for (auto &nm : names) {
    const uint64_t bytes = nm.count * es;
    const uint32_t src0 = (uint32_t)c.refs.size();
    for (uint32_t p : nm.prod) c.refs.push_back(ref_of(in_segs[p]));
    const uint32_t dst0 = (uint32_t)c.refs.size();
    for (uint32_t q : nm.cons) c.refs.push_back(ref_of(out_segs[q]));
    uint32_t piece = 0;
    for (uint64_t start = 0; start < bytes; start += U, ++piece) {
      coll_unit_t u;
      memset(&u, 0, sizeof(u));
      u.start = start;
      u.nbytes = (uint32_t)std::min<uint64_t>(U, bytes - start);
      u.src0 = src0;
      u.nsrc = (uint32_t)nm.prod.size();
      u.dst0 = dst0;
      u.ndst = (uint32_t)nm.cons.size();
      u.xoff = c.xpar_bytes;
      // tagged-data slots hold an epoch word beside every 4 payload bytes
      c.xpar_bytes += (uint64_t)u.nbytes * u.nsrc * (cfg.protocol == COLL_PROTO_LL ? 2u : 1u);
      u.pflag0 = c.n_pflag;
      c.n_pflag += u.nsrc;
      u.ncflag = twoshot ? 1u : u.ndst;
      u.cflag0 = c.n_cflag;
      c.n_cflag += u.ncflag;
      if (pull) {
        u.flags |= COLL_UNIT_PULL;
        u.roff = c.rpar_bytes;
        c.rpar_bytes += u.nbytes;
        u.dflag0 = c.n_dflag;
        c.n_dflag += u.ndst;
      }
      const uint32_t ui = (uint32_t)c.units.size();
      c.units.push_back(u);
      for (uint32_t j = 0; j < u.nsrc; ++j)
        S[in_segs[nm.prod[j]].rank].push_back(coll_item_t{ui, j});
      if (twoshot) {
        const uint32_t owner = (uint32_t)out_segs[nm.cons[piece % nm.cons.size()]].rank;
        C[owner].push_back(coll_item_t{ui, COLL_SLOT_ALL});
        if (pull)
          for (uint32_t i = 0; i < u.ndst; ++i)
            P[out_segs[nm.cons[i]].rank].push_back(coll_item_t{ui, i});
      } else {
        for (uint32_t i = 0; i < u.ndst; ++i)
          C[out_segs[nm.cons[i]].rank].push_back(coll_item_t{ui, i});
      }
    }
  }
  if (c.units.size() > 0x7FFFFFF0ull || c.n_pflag > 0x7FFFFFF0u || c.n_dflag > 0x7FFFFFF0u)
    return COLL_EINVAL;
  // warps: rank r gets W_r warps; item k of its stage (consume) list goes to warp k % W_r.
  // Every warp must be co-resident (they wait on each other), so the total is capped.
  std::vector<uint32_t> wbase(R + 1, 0);
  const uint32_t cap_r = std::max<uint32_t>(1u, (uint32_t)(max_warps > 0 ? max_warps : 1024) / (uint32_t)R);
  for (int r = 0; r < R; ++r) {
    uint32_t need = (uint32_t)std::max(std::max(S[r].size(), C[r].size()), P[r].size());
    uint32_t Wr = cfg.warps_per_rank ? std::min<uint32_t>(need, (uint32_t)cfg.warps_per_rank) : need;
    Wr = std::min(Wr, cap_r);
    wbase[r + 1] = wbase[r] + Wr;
  }
  const uint32_t nwarps = wbase[R];
  c.warps.resize(nwarps);
  std::vector<std::vector<uint32_t>> stage_of_warp(nwarps), cons_of_warp(nwarps),
      pull_of_warp(nwarps);
  for (int r = 0; r < R; ++r) {
    const uint32_t Wr = wbase[r + 1] - wbase[r];
    for (size_t k = 0; k < S[r].size(); ++k) stage_of_warp[wbase[r] + k % Wr].push_back((uint32_t)k);
    for (size_t k = 0; k < C[r].size(); ++k) cons_of_warp[wbase[r] + k % Wr].push_back((uint32_t)k);
    for (size_t k = 0; k < P[r].size(); ++k) pull_of_warp[wbase[r] + k % Wr].push_back((uint32_t)k);
  }
  // which warp stages / consumes each unit slot
  std::vector<std::vector<uint32_t>> stagers(c.units.size()), consumers(c.units.size());
  for (int r = 0; r < R; ++r) {
    const uint32_t Wr = wbase[r + 1] - wbase[r];
    for (uint32_t w = wbase[r]; w < wbase[r + 1]; ++w) {
      coll_warp_t &W = c.warps[w];
      memset(&W, 0, sizeof(W));
      W.rank = (uint32_t)r;
      W.rank_warps = Wr;
      W.s0 = (uint32_t)c.sitems.size();
      for (uint32_t k : stage_of_warp[w]) {
        c.sitems.push_back(S[r][k]);
        stagers[S[r][k].unit].push_back(w);
      }
      W.s1 = (uint32_t)c.sitems.size();
      W.c0 = (uint32_t)c.citems.size();
      for (uint32_t k : cons_of_warp[w]) {
        c.citems.push_back(C[r][k]);
        consumers[C[r][k].unit].push_back(w);
      }
      W.c1 = (uint32_t)c.citems.size();
      W.p0 = (uint32_t)c.pitems.size();
      for (uint32_t k : pull_of_warp[w]) c.pitems.push_back(P[r][k]);
      W.p1 = (uint32_t)c.pitems.size();
    }
  }
  // Dual buffers: restaging unit u (parity of epoch e) overwrites what u's consumers read
  // at epoch e-2. That is already ordered if every consumer warp of u notified epoch e-1
  // for a unit the stager consumed at e-1 (a consumer stages e-1 only after its e-2
  // consume, with release; the stager acquired that flag before restaging), or is the
  // stager itself. Otherwise the stager waits for the consumers' done flags explicitly.
  for (uint32_t ui = 0; ui < c.units.size(); ++ui) {
    coll_unit_t &u = c.units[ui];
    if (cfg.protocol == COLL_PROTO_BARRIER) {
      u.flags |= COLL_UNIT_DONE_FLAGS;
      continue;
    }
    bool implied = true;
    for (uint32_t P : stagers[ui]) {
      std::vector<uint32_t> seen;
      seen.push_back(P);
      const coll_warp_t &W = c.warps[P];
      for (uint32_t k = W.c0; k < W.c1; ++k)
        for (uint32_t w : stagers[c.citems[k].unit]) seen.push_back(w);
      std::sort(seen.begin(), seen.end());
      for (uint32_t Cw : consumers[ui])
        if (!std::binary_search(seen.begin(), seen.end(), Cw)) { implied = false; break; }
      if (!implied) break;
    }
    if (!implied) u.flags |= COLL_UNIT_REUSE_WAIT | COLL_UNIT_DONE_FLAGS;
  }
  *out = std::move(c);
  return COLL_OK;
}

void coll_fill_info(const coll_compiled &c, coll_plan_info_t *info) {
  if (!info) return;
  memset(info, 0, sizeof(*info));
  info->n_names = c.n_names;
  info->n_jobs = c.jobs.size();
  info->n_tiles = c.tiles.size();
  info->n_units = c.units.size();
  info->n_warps = c.warps.size();
  info->min_bytes = c.min_bytes;
  info->bulk_tile_bytes = c.bulk ? c.bulk_slot : 0;
  const bool dual = c.cfg.protocol != COLL_PROTO_BARRIER;
  info->xbuf_bytes = c.cfg.zero_copy ? 0 : (c.xpar_bytes + c.rpar_bytes) * (dual ? 2 : 1);
  info->flag_bytes = c.cfg.zero_copy ? 0
                                     : (uint64_t)c.n_pflag * 2 * 8 + (uint64_t)c.n_cflag * 4 +
                                           (uint64_t)c.units.size() * (c.rpar_bytes ? 2 * 4 : 0) +
                                           (uint64_t)c.n_dflag * 4;
}

extern "C" int coll_validate(int R, int op, int dtype, const coll_seg_t *in_segs, size_t n_in,
                             const uint64_t *in_len, const coll_seg_t *out_segs, size_t n_out,
                             const uint64_t *out_len, const coll_config_t *cfg,
                             coll_plan_info_t *info) {
  coll_compiled c;
  int e = coll_compile(R, op, dtype, in_segs, n_in, in_len, out_segs, n_out, out_len, cfg,
                       coll_default_max_warps(), coll_default_num_sms(), &c);
  if (e) return e;
  coll_fill_info(c, info);
  return COLL_OK;
}
