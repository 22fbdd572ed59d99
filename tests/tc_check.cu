// Host-only check of the tensor-core contraction's tables and constants
// (bit_expert_matvec_moe_b300/csrc/moe_tc.cuh), compiled and run by
// tests/test_plan_host.py.  For 4-bit and 2-bit rows of several widths it
// packs random canonical codes into the packed row layout (written here from
// the format description in moe_device.cuh, not from the pack kernel), takes
// every code stage the producer would copy (stage_code_x), unpacks each word
// with the field table the dequantising warps use (kField4 / kField2) through
// an fp16 emulation of the two fma steps, and checks that chunk position p of
// chunk c receives exactly code q of input 8c + chunk_perm(p).  It also checks
// the instruction and shared-memory descriptor encodings against hand-worked
// values, the swizzle's bijectivity and bank spread, and the shared-memory
// plan.  Prints "ok <checks>" and exits 0, or names the first violation.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "../bit_expert_matvec_moe_b300/csrc/moe_tc.cuh"

using namespace moe::tc;

namespace {

int g_checks = 0;
#define CHECK(cond, ...)                  \
  do {                                    \
    ++g_checks;                           \
    if (!(cond)) {                        \
      std::printf(__VA_ARGS__);           \
      std::printf("\n");                  \
      std::exit(1);                       \
    }                                     \
  } while (0)

float h2f(uint16_t bits) {
  __half_raw r;
  r.x = bits;
  return __half2float(__half(r));
}
uint16_t f2h_bits(double v) {  // round to nearest even, via float (exact for the values used here)
  const __half h = __float2half_rn((float)v);
  return __half_raw(h).x;
}

// one half of a field: fma(t, inv, neg) in fp16 (exact values here, so the
// fp16 rounding of the exact result is the hardware result)
double field_q(uint32_t w, const FieldSpec& f, int half) {
  const uint32_t t = ((w >> f.shift) & f.mask) | kMagic1024;
  const uint16_t tb = (uint16_t)(half ? t >> 16 : t & 0xFFFF);
  const uint16_t ib = (uint16_t)(half ? f.inv_m >> 16 : f.inv_m & 0xFFFF);
  const uint16_t nb = (uint16_t)(half ? f.neg_off >> 16 : f.neg_off & 0xFFFF);
  const double exact = (double)h2f(tb) * (double)h2f(ib) + (double)h2f(nb);
  return (double)h2f(f2h_bits(exact));
}

// packed code bytes of one row (format description in moe_device.cuh)
std::vector<uint8_t> pack_row(const std::vector<int>& q, int bits) {
  const int n_in = (int)q.size(), ng = n_in / 64;
  std::vector<uint8_t> row((size_t)n_in * bits / 8, 0);
  for (int g = 0; g < ng; ++g) {
    if (bits == 4) {
      const int k = g / 32, i = g % 32, n = std::min(32, ng - 32 * k);
      for (int h = 0; h < 2; ++h)
        for (int j = 0; j < 16; ++j) {
          const int in = 64 * g + 32 * h + 2 * j;
          row[1024 * k + 16 * (h * n + i) + j] = (uint8_t)(q[in] | (q[in + 1] << 4));
        }
    } else {
      for (int m = 0; m < 4; ++m)
        for (int j = 0; j < 4; ++j) {
          const int P[4] = {2 * j, 2 * j + 1, 8 + 2 * j, 9 + 2 * j};
          uint8_t b = 0;
          for (int t = 0; t < 4; ++t) b |= (uint8_t)(q[64 * g + 16 * m + P[t]] << (2 * t));
          row[16 * g + 4 * m + j] = b;
        }
    }
  }
  return row;
}

uint32_t word_at(const std::vector<uint8_t>& row, int off) {
  uint32_t w;
  std::memcpy(&w, row.data() + off, 4);
  return w;
}

void check_unpack(int bits, int n_in, unsigned seed) {
  std::srand(seed);
  std::vector<int> q(n_in);
  for (int& v : q) v = std::rand() % (1 << bits);
  const std::vector<uint8_t> row = pack_row(q, bits);
  const int ng = n_in / 64, nst = (ng + kStageGroups - 1) / kStageGroups;
  int groups_seen = 0;
  for (int st = 0; st < nst; ++st) {
    int x0, x1;
    stage_code_x(bits, ng, st, &x0, &x1);
    CHECK(x0 % 16 == 0 && x1 % 16 == 0, "stage %d: TMA x not 16-byte aligned", st);
    const int gcount = std::min(kStageGroups, ng - kStageGroups * st);
    for (int j = 0; j < gcount; ++j, ++groups_seen) {
      const int g = kStageGroups * st + j;
      for (int h = 0; h < 2; ++h) {
        // the 16 bytes (4-bit) or 8 bytes (2-bit) a dequantising thread reads
        const int base = bits == 4 ? (h ? x1 : x0) + 16 * j : x0 + 16 * j + 8 * h;
        CHECK(base + (bits == 4 ? 16 : 8) <= (int)row.size(), "piece outside the row's codes");
        const int nwords = bits == 4 ? 4 : 2;
        for (int m = 0; m < nwords; ++m) {
          const uint32_t w = word_at(row, base + 4 * m);
          const int nf = bits == 4 ? 4 : 8;
          for (int f = 0; f < nf; ++f) {
            const FieldSpec& fs = bits == 4 ? kField4[f] : kField2[f];
            // chunk and position this field fills
            const int c = bits == 4 ? 4 * h + m : 4 * h + 2 * m + f / 4;
            const int p0 = 2 * (f % 4);  // pair -> positions 2(f%4), 2(f%4)+1
            for (int half = 0; half < 2; ++half) {
              const int in = 64 * g + 8 * c + chunk_perm(p0 + half);
              const double got = field_q(w, fs, half);
              CHECK(got == (double)q[in], "bits %d n %d group %d half %d word %d field %d/%d: q %g, want %d (input %d)",
                    bits, n_in, g, h, m, f, half, got, q[in], in);
            }
          }
        }
      }
    }
  }
  CHECK(groups_seen == ng, "stages cover %d of %d groups", groups_seen, ng);
}

}  // namespace

int main() {
  // chunk order
  const int want_perm[8] = {0, 4, 1, 5, 2, 6, 3, 7};
  for (int p = 0; p < 8; ++p) CHECK(chunk_perm(p) == want_perm[p], "chunk_perm(%d)", p);

  // unpacking through the stages: several widths, chunks of 32 groups, ragged last stage
  const int widths[] = {64, 128, 256, 320, 512, 1024, 2048 + 64 * 5, 4096};
  unsigned seed = 1;
  for (int bits : {4, 2})
    for (int n_in : widths) check_unpack(bits, n_in, seed++);

  // fp16 constants
  CHECK(h2f(kMagic1024 & 0xFFFF) == 1024.f && h2f(kMagic1024 >> 16) == 1024.f, "magic 1024");
  CHECK(h2f(kOne & 0xFFFF) == 1.f && h2f(kM1024 & 0xFFFF) == -1024.f, "1, -1024");
  CHECK(h2f(kInv4 & 0xFFFF) == 0.25f && h2f(kM256 & 0xFFFF) == -256.f, "1/4, -256");
  CHECK(h2f(kInv16 & 0xFFFF) == 0.0625f && h2f(kM64 & 0xFFFF) == -64.f, "1/16, -64");
  CHECK(h2f(kInv64 & 0xFFFF) == 0.015625f && h2f(kM16 & 0xFFFF) == -16.f, "1/64, -16");

  // instruction descriptor: D f32 (bit 4), N >> 3 at bit 17, M >> 4 at bit 24
  CHECK(make_idesc_f16(128, 64) == 0x08100010u, "idesc 128x64: %08x", make_idesc_f16(128, 64));
  CHECK(make_idesc_f16(128, 16) == 0x08040010u, "idesc 128x16: %08x", make_idesc_f16(128, 16));
  CHECK(make_idesc_f16(128, 256) == 0x08400010u, "idesc 128x256: %08x", make_idesc_f16(128, 256));
  // shared-memory descriptor: start 0x1000 -> 0x100, LBO 16 -> 1 at bit 16,
  // SBO 1024 -> 64 at bit 32, version 1 at bit 46, swizzle 2 at bit 61
  CHECK(sdesc_sw128_kmajor(0x1000) == 0x4000404000010100ull, "sdesc: %016llx",
        (unsigned long long)sdesc_sw128_kmajor(0x1000));
  CHECK(sdesc_sw128_kmajor(0x1000 + 32) == sdesc_sw128_kmajor(0x1000) + 2, "descriptor advance of 32 bytes");

  // swizzle: a bijection of a 1024-byte atom; 8 consecutive rows at one chunk
  // hit 8 distinct 16-byte bank groups
  std::vector<int> seen(1024, 0);
  for (uint32_t r = 0; r < 8; ++r)
    for (uint32_t c = 0; c < 8; ++c) {
      const uint32_t o = swz128(r, c);
      CHECK(o < 1024 && o % 16 == 0 && !seen[o], "swizzle not a bijection at r %u c %u", r, c);
      seen[o] = 1;
    }
  for (uint32_t c = 0; c < 8; ++c) {
    int mask = 0;
    for (uint32_t r = 0; r < 8; ++r) mask |= 1 << ((swz128(r, c) % 128) / 16);
    CHECK(mask == 0xFF, "chunk %u: bank groups not spread", c);
  }

  // shared-memory plan
  CHECK(kOffCodes % 1024 == 0 && kKSlotBytes % 1024 == 0, "B slot alignment");
  CHECK(kTmemACol0 >= kDBufs * kDCols && kTmemACol0 + kKSlots * 32 <= kTmemCols, "A blocks after the accumulators");
  CHECK(kKSlots % 2 == 0, "even K ring: one writer per slot and lane quarter");
  CHECK(kCodeSlotBytes % 1024 == 0 && kHalfBoxBytes % 1024 == 0, "code box alignment");
  CHECK(kOffBars % 8 == 0 && kOffBars >= kOffCodes + kCodeSlots * kCodeSlotBytes, "barriers after the code slots");
  CHECK(kOffMisc + 12 <= kSmemUsed && kSmemBytes <= 232448, "plan total");
  CHECK(kBBytes == (uint32_t)(kTcTok / 8) * kBBoxBytes, "B slot holds kTcTok tokens of boxes");
  CHECK(2 * kTcTok <= kDCols && kTmemCols >= 32 && (kTmemCols & (kTmemCols - 1)) == 0, "tensor-memory columns");
  CHECK(kTcThreads == 32 * (kWarpDeq0 + 8) && kWarpEpi0 + 4 == kWarpDeq0, "warp roles");
  // epilogue and dequantising warps cover each tensor-memory lane quarter
  for (int qq = 0; qq < 4; ++qq) {
    int epi = 0, deq = 0;
    for (int w = kWarpEpi0; w < kWarpEpi0 + 4; ++w) epi += (w & 3) == qq;
    for (int w = kWarpDeq0; w < kWarpDeq0 + 8; ++w) deq += (w & 3) == qq;
    CHECK(epi == 1 && deq == 2, "lane quarter %d: %d epilogue, %d dequantising warps", qq, epi, deq);
  }
  std::printf("ok %d\n", g_checks);
  return 0;
}
