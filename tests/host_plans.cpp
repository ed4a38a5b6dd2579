// Host-side checks of the launch plans (no GPU): for every decode, Q8_1-decode,
// prefill and Q6_K plan over a grid of shapes, the tile and chunk counts stay in
// their documented ranges and the workspace offsets are 256-byte aligned, in
// order and inside the workspace. Built and run by test_host_plans.py.
#include <cstdio>

#include "kernels.h"

namespace {

int fails = 0;
#define CHECK(c, ...)                                               \
  do {                                                              \
    if (!(c)) {                                                     \
      if (++fails <= 20) {                                          \
        std::printf("FAIL line %d: %s: ", __LINE__, #c);            \
        std::printf(__VA_ARGS__);                                   \
        std::printf("\n");                                          \
      }                                                             \
    }                                                               \
  } while (0)

bool al(size_t o) { return o % 256 == 0; }

const int kDims[] = {256, 512, 768, 1024, 2048, 4096, 5120, 11008, 13824, 14336, 16384};

void check_decode(int sms) {
  for (int m = 1; m <= q4k::DECODE_PASS_MAX; ++m)
    for (int h : kDims)
      for (int i : kDims) {
        q4k::DecodePlan p;
        const bool ok = q4k::decode_plan(m, h, i, sms, &p);
        CHECK(ok, "m %d h %d i %d", m, h, i);
        if (!ok) continue;
        const int nt = (m + 3) / 4, max_nks = 16 / nt;
        CHECK(p.nt == nt, "m %d nt %d", m, p.nt);
        CHECK(p.nks1 >= 1 && p.nks1 <= max_nks && p.nks2 >= 1 && p.nks2 <= max_nks, "m %d h %d i %d nks %d %d", m, h,
              i, p.nks1, p.nks2);
        CHECK(p.kc1 >= 1 && p.kc2 >= 1 && p.grid1 >= 1 && p.grid2 >= 1, "m %d h %d i %d", m, h, i);
        const size_t offs[] = {p.off_fx1, p.off_fm1, p.off_sc1, p.off_fx2, p.off_fm2, p.off_sc2, p.off_p1, p.off_p2};
        for (int k = 0; k < 8; ++k) {
          CHECK(al(offs[k]), "m %d offset %d", m, k);
          if (k) CHECK(offs[k] > offs[k - 1], "m %d offsets %d", m, k);
        }
        CHECK(p.off_p1 + (size_t)p.nks1 * 2 * m * i * 4 <= p.off_p2, "m %d h %d i %d gate/up sums", m, h, i);
        CHECK(p.off_p2 + (size_t)p.nks2 * m * h * 4 <= p.ws_bytes, "m %d h %d i %d down sums", m, h, i);
        // x not in device memory (here: no device at all): K0 always runs
        CHECK(q4k::decode_kernels(p, false, 0, nullptr) == 4 + (p.nks2 > 1), "m %d kernels", m);
      }
  // the allocation-free entry point's static scratch holds every shape it accepts
  for (int m = 1; m <= q4k::NOALLOC_MAX_TOKENS; ++m)
    for (int h : kDims)
      for (int i : kDims) {
        if (h > q4k::NOALLOC_MAX_DIM || i > q4k::NOALLOC_MAX_DIM) continue;
        q4k::DecodePlan p;
        CHECK(q4k::decode_plan(m, h, i, sms, &p) && p.ws_bytes <= q4k::NOALLOC_SCRATCH_BYTES,
              "noalloc m %d h %d i %d: %zu bytes", m, h, i, p.ws_bytes);
      }
  q4k::DecodePlan p;
  // the GPU tests' many-chunk shapes (152 SMs): 8 gate/up chunks, 16 down chunks
  if (sms == 152) {
    CHECK(q4k::decode_plan(1, 16384, 256, sms, &p) && p.nks1 == 8, "m 1 h 16384 i 256 nks1 %d", p.nks1);
    CHECK(q4k::decode_plan(3, 16384, 256, sms, &p) && p.nks1 == 8, "m 3 h 16384 i 256 nks1 %d", p.nks1);
    CHECK(q4k::decode_plan(2, 256, 32768, sms, &p) && p.nks2 == 16, "m 2 h 256 i 32768 nks2 %d", p.nks2);
  }
  CHECK(!q4k::decode_plan(0, 4096, 11008, sms, &p), "m 0");
  CHECK(!q4k::decode_plan(q4k::DECODE_PASS_MAX + 1, 4096, 11008, sms, &p), "m above a pass");
}

void check_decode_q8(int sms) {
  for (int m = 1; m <= q4k::DECODE_PASS_MAX; ++m)
    for (int h : kDims)
      for (int i : kDims) {
        q4k::DecodeQ8Plan p;
        const bool ok = q4k::decode_q8_plan(m, h, i, sms, &p);
        CHECK(ok, "q8 m %d h %d i %d", m, h, i);
        if (!ok) continue;
        CHECK(p.fpath == (m > 2), "q8 m %d fpath %d", m, p.fpath);
        const size_t hq_bytes = (size_t)m * i + (size_t)m * (i / 32) * 8;
        CHECK(al(p.off_hq) && p.off_hq + hq_bytes <= p.ws_bytes, "q8 m %d hq", m);
        if (p.fpath) {
          CHECK(p.fp.m == m && p.fp.hidden == h && p.fp.inter == i, "q8 m %d embedded plan", m);
          CHECK(al(p.off_fp) && p.off_hq + hq_bytes <= p.off_fp && p.off_fp + p.fp.ws_bytes <= p.ws_bytes,
                "q8 m %d float-path workspace", m);
        } else {
          CHECK(p.mt >= m && p.mt <= 2, "q8 m %d mt %d", m, p.mt);
          CHECK(p.off_p2 + (size_t)p.nks2 * m * h * 4 <= p.ws_bytes, "q8 m %d down sums", m);
        }
      }
}

void check_prefill(int sms) {
  const int ms[] = {25, 64, 128, 129, 512, 2048, 4096};
  for (int m : ms)
    for (int h : kDims)
      for (int i : kDims) {
        q4k::PrefillPlan p;
        const bool ok = q4k::prefill_plan(m, h, i, sms, &p);
        CHECK(ok, "prefill m %d h %d i %d", m, h, i);
        if (!ok) continue;
        const int tiles = (h / 128) * ((m + 127) / 128);
        CHECK(p.ksplit >= 1 && p.ksplit <= 8, "m %d ksplit %d", m, p.ksplit);
        if (p.ksplit > 1) {
          CHECK(tiles * p.ksplit <= sms && p.tail_q == 0, "m %d h %d: K slices fill one round only", m, h);
          CHECK(i / 256 / p.ksplit >= 2, "m %d i %d: two superblocks per slice", m, i);
        }
        CHECK(p.tail_q == 0 || (p.tail_q >= 2 && p.tail_q <= 8), "m %d tail_q %d", m, p.tail_q);
        if (p.tail_q > 1) {
          const int ntail = tiles - p.tail_whole;
          CHECK(p.tail_whole > 0 && p.tail_whole % sms == 0 && ntail > 0 && ntail * p.tail_q <= sms,
                "m %d h %d: tail split %d %d", m, h, p.tail_whole, p.tail_q);
          CHECK(al(p.off_tail) && p.off_tail + (size_t)ntail * p.tail_q * 128 * 128 * 4 <= p.ws_bytes,
                "m %d h %d: tail scratch", m, h);
        }
        const int gtiles = (i / 64) * ((m + 127) / 128);
        CHECK(p.gu_q == 0 || (p.gu_q >= 2 && p.gu_q <= 8 && h / 256 / p.gu_q >= 2), "m %d h %d gu_q %d", m, h,
              p.gu_q);
        if (p.gu_q > 1) {
          const int ntail = gtiles - p.gu_whole;
          CHECK(p.gu_whole > 0 && p.gu_whole % sms == 0 && ntail > 0 && ntail * p.gu_q <= sms,
                "m %d i %d: gate/up tail split %d %d", m, i, p.gu_whole, p.gu_q);
          CHECK(al(p.off_gtail) && p.off_gtail + (size_t)ntail * p.gu_q * 128 * 128 * 4 <= p.ws_bytes,
                "m %d i %d: gate/up tail scratch", m, i);
        }
        const size_t offs[] = {p.off_xq, p.off_hq, p.off_xop, p.off_hop, p.off_misc, p.off_ypart};
        for (int k = 0; k < 6; ++k) CHECK(al(offs[k]) && offs[k] < p.ws_bytes, "m %d offset %d", m, k);
        CHECK(p.off_ypart + (size_t)p.ksplit * m * h * 4 <= p.ws_bytes, "m %d h %d partial outputs", m, h);
      }
  // the LLaMA-7B FFN at 64 tokens: 172 gate/up tiles on 152 SMs, the last 20 split in 7
  {
    q4k::PrefillPlan p7;
    CHECK(q4k::prefill_plan(64, 4096, 11008, 152, &p7) && p7.gu_whole == 152 && p7.gu_q == 7,
          "7B gate/up tail split %d %d", p7.gu_whole, p7.gu_q);
  }
  // the 27B-shaped long prefill: 640 down tiles on 152 SMs, the last 32 split in 4
  q4k::PrefillPlan p;
  CHECK(q4k::prefill_plan(2048, 5120, 17408, 152, &p) && p.ksplit == 1 && p.tail_whole == 608 && p.tail_q == 4,
        "27B prefill tail split %d %d", p.tail_whole, p.tail_q);
}

void check_q6k(int sms) {
  q4k::Q6Plan p;
  CHECK(q4k::q6k_plan(1, 32000, 4096, sms, &p) && p.grid >= 1 && al(p.off_fx) && al(p.off_sc) &&
            p.off_sc < p.ws_bytes,
        "q6k LM head");
  CHECK(!q4k::q6k_plan(9, 32000, 4096, sms, &p), "q6k m 9");
  CHECK(!q4k::q6k_plan(1, 32001, 4096, sms, &p), "q6k n not a multiple of 16");
}

}  // namespace

int main() {
  for (int sms : {152, 148, 132, 160, 170}) {
    check_decode(sms);
    check_decode_q8(sms);
    check_prefill(sms);
    check_q6k(sms);
  }
  std::printf(fails ? "%d failures\n" : "ok\n", fails);
  return fails ? 1 : 0;
}
