// Host-side check of the launch planner (rlca::make_plan in librlca.so),
// compiled and run by tests/test_planner_cpu.py without a GPU.  For a grid
// of estimators, sizes, layouts, storage types and pointer alignments it
// checks the invariants every driver relies on:
//   - rows and steps are covered: row_blocks * rows_per_cta >= E,
//     nseg * seg_len >= T > (nseg - 1) * seg_len, ntiles * tile >= T, and
//     segments are whole tiles;
//   - the fast drivers get only the shapes they assume (whole 4- or 8-step
//     chunks, one tile a row, 32-bit time-major offsets);
//   - CTAs are whole warps and fit the shared-memory limit;
//   - the workspace holds one affine map per (row, segment) when rows are
//     split, Retrace's per-step scalar planes after them, nothing otherwise;
//   - Retrace's time-major second pass (retrace_tail_plan) keeps the first
//     pass's segments in whole tiles of a fast time-major kernel that exists;
//   - tensor-copy tiles: each stage buffer starts on a 128-byte boundary,
//     the largest stage index a thread reads is the buffer's last element,
//     a box is at most 256 rows of whole 16-byte rows, the kernel's shared
//     memory fits, and the call's inputs permit the copies (E % 16 == 0).
// Prints "planner ok <plans checked>" with the number of plans of each
// driver, or the first failures; exit status 1 on any failure.
#include <cstdio>

#include "internal.h"
#include "rlca.h"

using namespace rlca;

namespace {

int g_bad = 0;

void fail(const char* what, int kind, long E, int T, unsigned flags, const Plan& p) {
  if (++g_bad <= 20)
    std::printf("FAIL %s: kind %d E=%ld T=%d flags=%#x width=%d env_width=%d tile=%d nseg=%d\n", what, kind, E, T,
                flags, p.width, p.env_width, p.tile, p.nseg);
}

template <class Est, int EW, int CT>
bool bulk_shape_ok(const Plan& p) {
  using S = TbShape<EW, CT>;
  using ST = typename Est::Store;
  bool ok = tb_smem_bytes<Est, EW, CT>() <= kMaxSmemPerCta;
  ok = ok && (S::FB * sizeof(ST)) % 128 == 0 && S::FBB % 128 == 0 && tb_stage_bytes<Est, EW, CT>() % 128 == 0;
  ok = ok && (CT - 1) * S::CS + (EW - 1) + (S::L - 1) * EW == S::FB - 1;
  // largest flag index: chunk CT - 1, our EW at offset FW - EW of the FW-wide copy, step L - 1
  ok = ok && (CT - 1) * S::L * S::FW + (S::FW - EW) + (EW - 1) + (S::L - 1) * S::FW == S::FBB - 1;
  ok = ok && S::TILE <= 256 && (EW * (int)sizeof(ST)) % 16 == 0 && S::FW % 16 == 0 && S::FW >= EW;
  ok = ok && p.tile == S::TILE && p.block == S::BLOCK;
  return ok;
}

template <class Est>
bool bulk_ok(const Plan& p) {
  if constexpr (sizeof(typename Est::Store) == 4) {
    if (p.env_width == 8) {
      switch (p.width) {
        case 4: return bulk_shape_ok<Est, 8, 4>(p);
        case 8: return bulk_shape_ok<Est, 8, 8>(p);
        case 16: return bulk_shape_ok<Est, 8, 16>(p);
        case 32: return bulk_shape_ok<Est, 8, 32>(p);
        default: return false;
      }
    }
  }
  if (p.env_width != 32) return false;
  switch (p.width) {
    case 1: return bulk_shape_ok<Est, 32, 1>(p);
    case 2: return bulk_shape_ok<Est, 32, 2>(p);
    case 4: return bulk_shape_ok<Est, 32, 4>(p);
    case 8: return bulk_shape_ok<Est, 32, 8>(p);
    default: return false;
  }
}

}  // namespace

int main() {
  const Kind kinds[] = {Kind::Gae, Kind::Disc, Kind::TdLambda, Kind::ValueTargets, Kind::Vtrace, Kind::Retrace,
                        Kind::Elig, Kind::PrefixSum, Kind::Affine};
  const long Es[] = {1, 3, 8, 33, 256, 1000, 1024, 4096, 9728, 9744, 16384, 65536};
  const int Ts[] = {1, 7, 8, 16, 31, 64, 128, 129, 256, 512, 520, 2048, 4096, 40000, 140001};
  const int sms = 152;
  long checked = 0, n_fast = 0, n_tm_fast = 0, n_staged = 0, n_bulk = 0, n_split = 0, n_tail = 0;
  for (int ki = 0; ki < 9; ++ki) {
    const Kind kind = kinds[ki];
    for (long E : Es)
      for (int T : Ts)
        for (unsigned layout : {0u, (unsigned)RLCA_TIME_MAJOR})
          for (unsigned extra : {0u, (unsigned)RLCA_BF16, (unsigned)RLCA_MULTIPASS})
            for (int align = 0; align < 3; ++align) {  // unaligned, 16-byte vectors, tensor-copy capable
              if ((extra & RLCA_BF16) && kind == Kind::PrefixSum) continue;
              if ((long long)E * T > (1ll << 31)) continue;
              const unsigned flags = layout | extra;
              const int A = kind == Kind::Retrace ? 18 : 0;
              const bool vec = align >= 1 && T % 4 == 0;
              const bool bulk = align == 2 && E % 16 == 0;
              Plan p;
              if (!make_plan(kind, E, T, A, flags, sms, vec, &p, bulk)) {
                fail("no plan", ki, E, T, flags, p);
                continue;
              }
              ++checked;
              n_fast += p.fast;
              n_tm_fast += p.tm_fast;
              n_staged += p.tm_staged;
              n_bulk += p.tm_bulk;
              n_split += p.nseg > 1;
              const bool tm = (flags & RLCA_TIME_MAJOR) != 0;
              if (p.time_major != tm) fail("layout", ki, E, T, flags, p);
              if (p.block <= 0 || p.block > 1024 || (p.block % 32 != 0 && p.block != p.width))
                fail("block", ki, E, T, flags, p);
              if ((long long)p.row_blocks * p.rows_per_cta < E) fail("rows covered", ki, E, T, flags, p);
              if ((long long)p.nseg * p.seg_len < T || (long long)(p.nseg - 1) * p.seg_len >= T)
                fail("segments cover T", ki, E, T, flags, p);
              if (p.seg_len % p.tile != 0) fail("segment of whole tiles", ki, E, T, flags, p);
              if ((long long)p.ntiles * p.tile < T || (long long)(p.ntiles - 1) * p.tile >= T)
                fail("tiles cover T", ki, E, T, flags, p);
              if (p.fast && (tm || !vec || p.nseg != 1 || T % p.steps != 0 || p.width * p.steps != p.tile ||
                             p.tile < T || p.rows_per_cta * p.width != p.block))
                fail("env-major fast driver", ki, E, T, flags, p);
              if (p.tm_fast && (!tm || T % 8 != 0 || (unsigned long long)E * T >= (1ull << 32) ||
                                p.block != p.env_width * p.width || p.tile != 8 * p.width || p.block % 32 != 0))
                fail("time-major fast driver", ki, E, T, flags, p);
              if ((p.tm_staged || p.tm_bulk) && !p.tm_fast) fail("staged without the fast driver", ki, E, T, flags, p);
              if (p.smem + p.smem_driver_bound > kMaxSmemPerCta) fail("shared memory", ki, E, T, flags, p);
              const size_t map = kind == Kind::ValueTargets ? 16 : 8;
              if (p.nseg > 1) {
                if (p.ws_bytes < (size_t)E * p.nseg * map) fail("workspace maps", ki, E, T, flags, p);
                if (kind == Kind::Retrace &&
                    (p.aux_bytes != (size_t)12 * E * T || p.ws_bytes < p.aux_bytes + (size_t)E * p.nseg * 8 ||
                     aux_offset(p.ws_bytes, p.aux_bytes) % 256 != 0))
                  fail("Retrace scalar planes", ki, E, T, flags, p);
              } else if (p.ws_bytes != 0) {
                fail("workspace without a split", ki, E, T, flags, p);
              }
              if (kind == Kind::Retrace) {
                Plan q;
                const bool b16 = (flags & RLCA_BF16) != 0;
                if (retrace_tail_plan(p, E, T, b16, &q)) {
                  ++n_tail;
                  const int EW = b16 ? 16 : 8;
                  const bool widths = b16 ? (q.width >= 2 && q.width <= 32) : (q.width >= 4 && q.width <= 32);
                  if (!tm || p.nseg < 2 || T % 8 != 0 || (unsigned long long)E * T >= (1ull << 32) ||
                      q.env_width != EW || !widths || (q.width & (q.width - 1)) != 0 || q.block != EW * q.width ||
                      q.block % 32 != 0 || q.tile != 8 * q.width || q.seg_len != p.seg_len || q.nseg != p.nseg ||
                      q.seg_len % q.tile != 0 || (long long)q.row_blocks * EW < E || !q.tm_fast || q.tm_staged ||
                      q.tm_bulk || q.smem + q.smem_driver_bound > kMaxSmemPerCta)
                    fail("Retrace second pass", ki, E, T, flags, q);
                } else if (tm && p.nseg > 1 && T % 8 == 0 && (unsigned long long)E * T < (1ull << 32)) {
                  fail("Retrace second pass not taken", ki, E, T, flags, p);
                }
              }
              if (p.tm_bulk) {
                const bool b16 = (flags & RLCA_BF16) != 0;
                bool ok = bulk && tm && E % 16 == 0 && T % 8 == 0 &&
                          (p.env_width == 32 ? E >= 64L * sms
                                             : (p.env_width == 8 && !b16 && E < 64L * sms && p.nseg == 1 &&
                                                p.ntiles >= 4));
                switch (kind) {
                  case Kind::Gae: ok = ok && (b16 ? bulk_ok<GaeEst<true, bf16>>(p) : bulk_ok<GaeEst<true>>(p)); break;
                  case Kind::ValueTargets:
                    ok = ok && (b16 ? bulk_ok<ValueTargetsEst<true, bf16>>(p) : bulk_ok<ValueTargetsEst<true>>(p));
                    break;
                  case Kind::Vtrace:
                    ok = ok && (b16 ? bulk_ok<VtraceEst<true, bf16>>(p) : bulk_ok<VtraceEst<true>>(p));
                    break;
                  case Kind::Retrace: ok = false; break;
                  default: break;
                }
                if (!ok) fail("tensor-copy tiles", ki, E, T, flags, p);
              }
            }
  }
  if (g_bad != 0) {
    std::printf("planner: %d failures in %ld plans\n", g_bad, checked);
    return 1;
  }
  std::printf("planner ok %ld fast %ld tm_fast %ld staged %ld bulk %ld two_pass %ld retrace_tail %ld\n", checked,
              n_fast, n_tm_fast, n_staged, n_bulk, n_split, n_tail);
  return 0;
}
