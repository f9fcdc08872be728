"""The K-grouped kernel's issue order (csrc/kgemm_plan.cuh), compiled as plain
C++ on the host and walked for every worker over many group-size
distributions -- skewed, uniform, empty and one-row experts, experts of one
and of several accumulation chunks, one expert, 1024 experts -- in tile and
chunk mode, with several row-block, chunk and light-expert sizes.  For each
walk it checks that
  * every item of the list is walked by exactly one worker (i = worker mod W)
    and every row block of every chunk of it exactly once, in row order, the
    blocks of one accumulator contiguous in its own stream, with the first
    and last block flagged; an item of an expert without rows gets on_zero
    and no block;
  * an accumulator never starts in a buffer whose previous accumulator has
    not ended, and the parity of each use of a buffer alternates -- which is
    what the MMA issuer and the epilogue rely on not to wait on each other
    forever; with both buffers free it takes the one whose last accumulator
    ended first (the first the epilogue frees);
  * heavy items are walked in list order, light ones in list order, and light
    item j starts after exactly floor(j HB / L) heavy row blocks;
  * the walk's segments -- runs of row blocks of one accumulator, which the
    kernel's roles loop over -- are whole blocks of one chunk, the first one
    starting its accumulator and only the last one ending it, and a light
    item is one segment;
  * a walk stopped by a callback returns false at once."""
import shutil
import subprocess

import pytest

from moe_grouped_gemm_device_gb300 import _build

PROGRAM = r"""
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <random>
#include <vector>
#include "kgemm_plan.cuh"
using namespace rg::kgplan;

static long fails = 0, walks = 0, blocks_total = 0;
#define CHECK(c, ...) do { if (!(c)) { if (fails < 20) { std::printf("FAILED %s: ", #c); \
  std::printf(__VA_ARGS__); std::printf("\n"); } ++fails; } } while (0)

struct Case { std::vector<int> counts; int tpe, nworkers; bool chunked; int br, chunk, light; const char* what; };

static void run_case(const Case& cs) {
  const int E = (int)cs.counts.size();
  std::vector<int> off(E + 1, 0), ord(E), up(E + 1, 0), pos(E);
  for (int e = 0; e < E; ++e) off[e + 1] = off[e] + cs.counts[e];
  for (int e = 0; e < E; ++e) ord[e] = e;
  std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return cs.counts[a] > cs.counts[b]; });
  for (int p = 0; p < E; ++p) pos[ord[p]] = p;
  const Tables t{off.data(), ord.data(), up.data(), E, cs.tpe, cs.chunked, cs.chunk};
  for (int p = 0; p < E; ++p) up[p + 1] = up[p] + t.nchunks(ord[p]) * cs.tpe;
  const int NI = t.items();
  std::vector<int> item_seen(NI, 0);
  // chunks of item i completed (bit mask is enough: at most 2^20 rows / chunk)
  std::vector<long long> chunk_done(NI, 0);
  for (int w = 0; w < cs.nworkers; ++w) {
    const Plan p = make_plan(t, w, cs.nworkers, cs.br, cs.light);
    ++walks;
    int open_item[2] = {-1, -1}, open_chunk[2] = {-1, -1}, next_r[2] = {0, 0};
    unsigned uses[2] = {0, 0};
    long end_seq[2] = {-1, -1}, ends = 0;  // when each buffer's last accumulator ended
    int hb = 0, lights = 0, last_heavy = -1, last_light = -1, items = 0, cur_heavy = -1, cur_chunk = -1;
    auto note_item = [&](int i, bool light) {
      CHECK(i >= 0 && i < NI, "%s: item %d of %d", cs.what, i, NI);
      if (i < 0 || i >= NI) return;
      CHECK(i % cs.nworkers == w, "%s: item %d walked by worker %d", cs.what, i, w);
      CHECK(item_seen[i] == 0, "%s: item %d walked twice", cs.what, i);
      item_seen[i] = 1;
      ++items;
      if (light) {
        CHECK(i > last_light, "%s: light item %d after %d", cs.what, i, last_light);
        // light item j starts after floor(j HB / L) heavy blocks
        const long long want = p.HB ? (long long)lights * p.HB / p.L : 0;
        CHECK(hb == want, "%s: light %d of %d after %d heavy blocks, not %lld (HB %d)", cs.what, lights, p.L, hb,
              want, p.HB);
        last_light = i;
        ++lights;
      } else {
        CHECK(i > last_heavy, "%s: heavy item %d after %d", cs.what, i, last_heavy);
        last_heavy = i;
      }
    };
    const bool ok = walk_blocks(t, p,
      [&](const Item& it, int c, int cs_, int ce, int r, Acc a, bool first, bool last) {
        ++blocks_total;
        const int e = it.e;
        const bool light = t.rows(e) < cs.light;
        const int i = t.chunked ? up[pos[e]] + it.c0 * t.tpe + it.local : pos[e] * t.tpe + it.local;
        CHECK(c >= it.c0 && c < it.c1, "%s: chunk %d outside [%d, %d)", cs.what, c, it.c0, it.c1);
        CHECK(cs_ == off[e] + c * t.chunk_rows && ce == std::min(off[e + 1], cs_ + t.chunk_rows) && cs_ < ce,
              "%s: chunk rows [%d, %d) of expert %d chunk %d", cs.what, cs_, ce, e, c);
        CHECK(a.buf == 0 || a.buf == 1, "%s: buffer %d", cs.what, a.buf);
        if (first) {
          CHECK(r == cs_, "%s: first block at %d, chunk starts at %d", cs.what, r, cs_);
          CHECK(open_item[a.buf] < 0, "%s: accumulator of item %d starts in buffer %d still open for item %d",
                cs.what, i, a.buf, open_item[a.buf]);
          CHECK(a.par == (uses[a.buf] & 1u), "%s: parity %u of use %u of buffer %d", cs.what, a.par, uses[a.buf],
                a.buf);
          // with the other buffer free too, the one whose last accumulator ended first
          CHECK(open_item[1 - a.buf] >= 0 || end_seq[a.buf] <= end_seq[1 - a.buf],
                "%s: item %d takes buffer %d (last end %ld), not %d (last end %ld)", cs.what, i, a.buf,
                end_seq[a.buf], 1 - a.buf, end_seq[1 - a.buf]);
          ++uses[a.buf];
          open_item[a.buf] = i;
          open_chunk[a.buf] = c;
          next_r[a.buf] = cs_;
          if (light || i != cur_heavy) {  // a new item (its first chunk)
            note_item(i, light);
            CHECK(c == it.c0, "%s: item %d starts at chunk %d, not %d", cs.what, i, c, it.c0);
            CHECK(!light || it.c1 == it.c0 + 1, "%s: light item %d of several chunks", cs.what, i);
            if (!light) {
              CHECK(cur_heavy < 0 || chunk_done[cur_heavy] >> (cur_chunk) & 1, "%s: heavy item %d left at chunk %d",
                    cs.what, cur_heavy, cur_chunk);
              cur_heavy = i;
            }
          } else {
            CHECK(c == cur_chunk + 1, "%s: item %d chunk %d after %d", cs.what, i, c, cur_chunk);
          }
          if (!light) cur_chunk = c;
          // a light accumulator starts only between heavy row blocks: the open
          // heavy accumulator (if any) holds the other buffer
          if (light) CHECK(open_item[1 - a.buf] < 0 || open_item[1 - a.buf] != i, "%s: item %d in both buffers",
                           cs.what, i);
        }
        CHECK(open_item[a.buf] == i && open_chunk[a.buf] == c, "%s: block of item %d chunk %d in buffer %d of "
              "item %d chunk %d", cs.what, i, c, a.buf, open_item[a.buf], open_chunk[a.buf]);
        CHECK(r == next_r[a.buf], "%s: block at %d, expected %d", cs.what, r, next_r[a.buf]);
        next_r[a.buf] = r + p.br;
        CHECK(last == (r + p.br >= ce), "%s: last flag at %d of [%d, %d)", cs.what, r, cs_, ce);
        if (!light) ++hb;
        if (last) {
          open_item[a.buf] = -1;
          end_seq[a.buf] = ends++;
          if (i >= 0 && i < NI) {
            CHECK(!(chunk_done[i] >> c & 1), "%s: chunk %d of item %d twice", cs.what, c, i);
            chunk_done[i] |= 1ll << c;
          }
        }
        return true;
      },
      [&](const Item& it) {
        CHECK(t.rows(it.e) == 0, "%s: on_zero for expert %d of %d rows", cs.what, it.e, t.rows(it.e));
        const int i = t.chunked ? up[pos[it.e]] + it.c0 * t.tpe + it.local : pos[it.e] * t.tpe + it.local;
        note_item(i, true);
        return true;
      });
    CHECK(ok, "%s: walk returned false", cs.what);
    // the segments: each a run of whole row blocks of one accumulator, the
    // first starting the accumulator and only the last ending it; a heavy
    // segment stops at its accumulator's end or just before a light item
    {
      bool in_heavy = false;
      walk(t, p, [&](const Item& it, int, int cs_, int ce, int r0, int r1, Acc, bool first, bool last) {
        const bool light = t.rows(it.e) < cs.light;
        CHECK(r0 < r1 && (r0 - cs_) % p.br == 0 && first == (r0 == cs_) && last == (r1 == ce) &&
              (last || (r1 - cs_) % p.br == 0), "%s: segment [%d, %d) of chunk [%d, %d) first %d last %d",
              cs.what, r0, r1, cs_, ce, first, last);
        CHECK(!light || (first && last), "%s: light item in several segments", cs.what);
        if (!light) in_heavy = !last;
        return true; }, [&](const Item&) { return true; });
      CHECK(!in_heavy, "%s: heavy accumulator left open by the segments", cs.what);
    }
    CHECK(open_item[0] < 0 && open_item[1] < 0, "%s: accumulator left open", cs.what);
    CHECK(hb == p.HB, "%s: %d heavy blocks walked, plan says %d", cs.what, hb, p.HB);
    CHECK(items == p.n_items && lights == p.L, "%s: %d items (%d light), plan %d (%d)", cs.what, items, lights,
          p.n_items, p.L);
    // a callback that stops the walk
    int calls = 0;
    const int stop_at = p.n_items ? 1 + (w % 5) : 0;
    const bool r2 = walk_blocks(t, p, [&](const Item&, int, int, int, int, Acc, bool, bool) {
                           return ++calls < stop_at; }, [&](const Item&) { return ++calls < stop_at; });
    if (p.n_items) {
      const bool stopped = !r2;
      CHECK(stopped ? calls == stop_at : calls < stop_at, "%s: stopped walk made %d calls (stop at %d)", cs.what,
            calls, stop_at);
    }
  }
  for (int i = 0; i < NI; ++i) {
    CHECK(item_seen[i] == 1, "%s: item %d walked %d times", cs.what, i, item_seen[i]);
    const int e = t.chunked ? -1 : ord[i / t.tpe];
    if (!t.chunked && t.rows(e) > 0) {
      const long long all = (1ll << t.nchunks(e)) - 1;
      CHECK(chunk_done[i] == all, "%s: item %d chunks %llx of %llx", cs.what, i, chunk_done[i], all);
    }
    if (t.chunked) {
      int p = 0;
      while (up[p + 1] <= i) ++p;
      if (t.rows(ord[p]) > 0) {
        const int c = (i - up[p]) / t.tpe;
        CHECK(chunk_done[i] == (1ll << c), "%s: chunk item %d done %llx", cs.what, i, chunk_done[i]);
      }
    }
  }
}

int main() {
  std::mt19937 rng(12345);
  std::vector<Case> cases;
  auto zipf = [&](int E, int M, double s) {
    std::vector<double> w(E);
    for (int e = 0; e < E; ++e) w[e] = 1.0 / std::pow(e + 1.0, s);
    std::shuffle(w.begin(), w.end(), rng);
    double sum = 0; for (double x : w) sum += x;
    std::vector<int> c(E); int tot = 0;
    for (int e = 0; e < E; ++e) { c[e] = (int)(w[e] / sum * M); tot += c[e]; }
    c[0] += M - tot;
    return c;
  };
  auto uni = [&](int E, int lo, int hi) {
    std::vector<int> c(E); std::uniform_int_distribution<int> d(lo, hi);
    for (int& x : c) x = d(rng);
    return c;
  };
  std::vector<std::vector<int>> dists = {
    zipf(128, 65536, 1.2), zipf(32, 32768, 0.8), zipf(7, 40000, 1.5), uni(32, 0, 2000), uni(64, 0, 300),
    uni(1024, 0, 5), {9000, 0, 37, 4100, 8192, 4032, 4033, 1, 12000}, {20000, 130, 0, 16200, 7, 4032},
    {0, 0, 0}, {1}, {4032}, {96, 192, 95, 97, 0, 511, 512, 513}, {17725}, std::vector<int>(40, 1000),
  };
  for (size_t d = 0; d < dists.size(); ++d)
    for (int tpe : {1, 2, 20, 60, 81, 120})
      for (int nw : {76, 7, 1})
        for (int chunked = 0; chunked < 2; ++chunked)
          for (int light : {1, 512, 4032}) {
            cases.push_back({dists[d], tpe, nw, chunked != 0, 96, 4032, light, "br96"});
            if (light == 512) cases.push_back({dists[d], tpe, nw, chunked != 0, 128, 4096, 1000, "br128"});
          }
  for (const Case& c : cases) run_case(c);
  std::printf("%ld walks, %ld blocks, %ld failures\n", walks, blocks_total, fails);
  std::printf("%s\n", fails ? "SOME CHECKS FAILED" : "ALL CHECKS PASSED");
  return fails != 0;
}
"""


@pytest.mark.skipif(shutil.which("g++") is None, reason="g++ not available")
def test_kgemm_issue_order_on_the_host(tmp_path):
    src = tmp_path / "plan_test.cc"
    src.write_text(PROGRAM)
    exe = tmp_path / "plan_test"
    r = subprocess.run(["g++", "-std=c++17", "-O2", "-I", _build.CSRC, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ALL CHECKS PASSED" in r.stdout, r.stdout
