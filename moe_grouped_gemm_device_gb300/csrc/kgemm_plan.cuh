// Issue order of the K-grouped weight-gradient kernel's persistent workers:
// which tile (and row chunk) each worker computes, in which order its row
// blocks go through the shared-memory ring, and which tensor-memory buffer
// each accumulator uses.  The producers, the MMA issuer and the epilogue of a
// CTA all run walk() over the same tables, so they agree on all three by
// construction.  Plain host/device code: the host tests run it over many
// group-size distributions and check its invariants.
#pragma once

#include <cstdint>

#ifndef RG_HD
#if defined(__CUDACC__)
#define RG_HD __host__ __device__ __forceinline__
#else
#define RG_HD inline
#endif
#endif

namespace rg {
namespace kgplan {

RG_HD int imin(int a, int b) { return a < b ? a : b; }
RG_HD int imax(int a, int b) { return a > b ? a : b; }

// The expert tables of a launch (shared memory in the kernel).
struct Tables {
  const int* off;   // [E+1] row offsets of the experts
  const int* ord;   // [E] experts by decreasing row count, ties by index
  const int* up;    // [E+1] chunk mode: first item of each position of ord, up[E] = items
  int E;
  int tpe;          // dW tiles per expert
  bool chunked;     // items are single row chunks of a tile (else whole tiles)
  int chunk_rows;   // rows of an expert summed in one accumulator

  RG_HD int rows(int e) const { return off[e + 1] - off[e]; }
  RG_HD int nchunks(int e) const { return imax(1, (rows(e) + chunk_rows - 1) / chunk_rows); }
  RG_HD int items() const { return chunked ? up[E] : E * tpe; }
};

// Item i of the list: expert e, its tile `local`, row chunks [c0, c1) of nch.
// Tile mode: item i is tile i of the list of E x tpe tiles, experts in the
// order `ord`, with all of its chunks.  Chunk mode: the items of the expert
// at position p of `ord` are up[p] .. up[p+1]-1, chunk by chunk (chunk 0 of
// every tile, then chunk 1, ...).
struct Item {
  int e, local, c0, c1, nch;
};

// `pe` is the caller's position in `ord`, advanced as i grows (chunk mode);
// start it at 0 and call with non-decreasing i.
RG_HD Item item_at(const Tables& t, int i, int& pe) {
  Item it;
  if (t.chunked) {
    while (t.up[pe + 1] <= i) ++pe;
    const int j = i - t.up[pe];
    it.e = t.ord[pe];
    it.c0 = j / t.tpe;
    it.c1 = it.c0 + 1;
    it.local = j - it.c0 * t.tpe;
  } else {
    pe = i / t.tpe;
    it.e = t.ord[pe];
    it.local = i - pe * t.tpe;
    it.c0 = 0;
    it.c1 = t.nchunks(it.e);
  }
  it.nch = t.nchunks(it.e);
  return it;
}

// One worker's share.  Its items are i = worker + k * nworkers, k = 0 ..
// n_items-1.  An item of an expert with fewer than light_rows rows is light:
// storing its dW tile takes longer than its MMAs.  The list is longest first,
// so the first nh items (HB row blocks in all) are heavy and the L others
// light.
struct Plan {
  int worker, nworkers;
  int n_items, nh, L, HB;
  int br;  // rows per row block (stage)
};

RG_HD Plan make_plan(const Tables& t, int worker, int nworkers, int br, int light_rows) {
  Plan p;
  p.worker = worker;
  p.nworkers = nworkers;
  p.br = br;
  const int NI = t.items();
  p.n_items = worker < NI ? (NI - worker + nworkers - 1) / nworkers : 0;
  int heavy = 0;  // experts with at least light_rows rows: a prefix of ord (binary search)
  for (int top = t.E; heavy < top;) {
    const int mid = (heavy + top) >> 1;
    if (t.rows(t.ord[mid]) >= light_rows) heavy = mid + 1;
    else top = mid;
  }
  const int G = t.chunked ? t.up[heavy] : heavy * t.tpe;  // first light item of the list
  p.nh = G > worker ? imin(p.n_items, (G - worker + nworkers - 1) / nworkers) : 0;
  p.L = p.n_items - p.nh;
  p.HB = 0;
  int pe = 0;
  for (int k = 0; k < p.nh; ++k) {
    const Item it = item_at(t, worker + k * nworkers, pe);
    const int rb = t.off[it.e], re = t.off[it.e + 1];
    for (int c = it.c0; c < it.c1; ++c)
      p.HB += (imin(re, rb + (c + 1) * t.chunk_rows) - rb - c * t.chunk_rows + br - 1) / br;
  }
  return p;
}

// An accumulator: tensor-memory buffer 0 or 1, and the parity of this use of
// the buffer (uses of a buffer alternate between filling and draining).
struct Acc {
  int buf;
  uint32_t par;
};

// The worker's issue order.  Issued in list order, the heavy items would keep
// the tensor cores busy while the epilogue waits, and the light items' stores
// would then run with the tensor cores idle.  Instead light item j is issued
// whole between two row blocks of the heavy sequence, before heavy block
// floor(j HB / L), so that its stores overlap heavy MMAs.  A light
// accumulator started while a heavy one is open takes the other buffer; every
// other accumulator takes the buffer whose last accumulator ended first.  So
// an accumulator never starts in a buffer whose previous accumulator has not
// ended (been committed), and the epilogue, which drains accumulators in the
// order they end, can always free the buffer the next one waits for.
//
// The walk goes segment by segment: a segment is a run of consecutive row
// blocks r0, r0 + br, ... < r1 of one accumulator -- a whole light item, or a
// heavy accumulator's blocks up to its end or to the next light item's place
// (heavy block floor(j HB / L)), whichever comes first -- so that the roles
// loop over the blocks of a segment with nothing else to decide.
// on_segment(item, chunk c, chunk rows [cs, ce), r0, r1, acc, first segment
// of the accumulator (r0 == cs), last segment (r1 == ce)) is called for every
// segment in issue order; on_zero(item) for an item of an expert without rows
// (no MMA, no accumulator), at its place among the light items.  Either
// returning false stops the walk, which then returns false.
template <class OnSegment, class OnZero>
RG_HD bool walk(const Tables& t, const Plan& p, OnSegment&& on_segment, OnZero&& on_zero) {
  const int br = p.br;
  int kh = 0, kl = p.nh, hb = 0, pe_h = 0, pe_l = 0;
  int last_buf = 1, hbuf = 0;
  uint32_t uses0 = 0, uses1 = 0;  // accumulators begun in each buffer
  bool hopen = false;
  auto begin_acc = [&](bool light) {
    Acc a;
    a.buf = (light && hopen) ? 1 - hbuf : 1 - last_buf;
    a.par = (a.buf ? uses1++ : uses0++) & 1u;
    if (!light) {
      hopen = true;
      hbuf = a.buf;
    }
    return a;
  };
  Item hi{};
  int hc = 0, hcs = 0, hce = 0, hr = 0;  // heavy item: chunk, its rows [hcs, hce), next row block
  auto heavy_item = [&](int k) {
    hi = item_at(t, p.worker + k * p.nworkers, pe_h);
    hc = hi.c0;
    hcs = t.off[hi.e] + hc * t.chunk_rows;
    hce = imin(t.off[hi.e + 1], hcs + t.chunk_rows);
    hr = hcs;
  };
  if (p.nh > 0) heavy_item(0);
  // the heavy block before which light item kl is issued: floor(j HB / L), j = kl - nh
  auto light_due = [&]() {
    return kl < p.n_items ? static_cast<int>(static_cast<long long>(kl - p.nh) * p.HB / p.L) : 0;
  };
  int due = light_due();
  Acc ha{0, 0u};
  while (true) {
    if (kl < p.n_items && (kh >= p.nh || hb >= due)) {
      const Item li = item_at(t, p.worker + kl * p.nworkers, pe_l);
      ++kl;
      due = light_due();
      const int rb = t.off[li.e], re = t.off[li.e + 1];
      if (rb == re) {
        if (!on_zero(li)) return false;
        continue;
      }
      const Acc a = begin_acc(true);
      if (!on_segment(li, 0, rb, re, rb, re, a, true, true)) return false;
      last_buf = a.buf;
      continue;
    }
    if (kh >= p.nh) break;
    const bool first = hr == hcs;
    if (first) ha = begin_acc(false);
    // here due > hb: the next light item, if any, comes after at least one block
    const int left = (hce - hr + br - 1) / br;
    const int step = kl < p.n_items ? imin(left, due - hb) : left;
    const bool last = step == left;
    const int r1 = last ? hce : hr + step * br;
    if (!on_segment(hi, hc, hcs, hce, hr, r1, ha, first, last)) return false;
    hb += step;
    hr = r1;
    if (last) {
      last_buf = ha.buf;
      hopen = false;
      if (++hc < hi.c1) {
        hcs = hce;
        hce = imin(t.off[hi.e + 1], hcs + t.chunk_rows);
        hr = hcs;
      } else if (++kh < p.nh) {
        heavy_item(kh);
      }
    }
  }
  return true;
}

// The same walk block by block: on_block(item, chunk c, chunk rows [cs, ce),
// row block start r, acc, first block of the accumulator, last block).
template <class OnBlock, class OnZero>
RG_HD bool walk_blocks(const Tables& t, const Plan& p, OnBlock&& on_block, OnZero&& on_zero) {
  return walk(
      t, p,
      [&](const Item& it, int c, int cs, int ce, int r0, int r1, Acc a, bool, bool last) {
        for (int r = r0; r < r1; r += p.br)
          if (!on_block(it, c, cs, ce, r, a, r == cs, last && r + p.br >= r1)) return false;
        return true;
      },
      on_zero);
}

}  // namespace kgplan
}  // namespace rg
