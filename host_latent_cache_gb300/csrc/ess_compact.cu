// Compact 656-byte latent rows (host code only).
//
// "ESS: Latent-Cache Offload" (foosynaptic tech notes): the latent entry is
// c^KV[512] + k^R[64]; the page quotes host transfers of about 656 bytes
// (its table of mechanisms, the FlashTrans + UVA row) and splits per-token
// bytes 16.8% indexer / 83.2% latent, which 132 and 656 bytes give exactly.
// The layout is a reading (656 = 512 + 16 + 128): the 512 latent values as
// e4m3 in four tiles of 128, one float32 scale per tile, then the 64 RoPE
// values as bf16.
//
// A tile's scale is the smallest power of two at or above amax / 448 in float32
// (1 for an all-zero tile), 448 being the largest finite e4m3 value; a power
// of two so that every decoded value is exact in bf16.  A value's code is its
// (exact) quotient by the scale rounded to the nearest e4m3 value, ties to the
// even code, saturating at 448, the sign kept.  The e4m3 format: 1 sign bit, 4 exponent
// bits with bias 7, 3 mantissa bits; exponent 0 holds the subnormals m * 2^-9;
// the code with all exponent and mantissa bits set is NaN, so 448 (exponent
// 15, mantissa 6) is the largest finite value.
#include <cmath>
#include <cstring>

#include "ess_internal.h"

namespace {

constexpr int kTile = 128;
constexpr int kTiles = ess::kLatent / kTile;
constexpr int kCompactBytes = ess::kLatent + 4 * kTiles + 2 * (ess::kRowDim - ess::kLatent);

float bf16_to_float(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

uint8_t e4m3_encode(float q) {
  const uint8_t sign = std::signbit(q) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(q));
  if (!(a < 448.0)) return sign | 0x7E;               // saturate (and NaN input)
  if (a < 0x1p-6) {                                     // subnormal range: m * 2^-9
    const double m = std::nearbyint(a * 512.0);         // ties to even; 8 becomes 2^-6
    return sign | static_cast<uint8_t>(m);
  }
  int e;
  const double fr = std::frexp(a, &e);                  // a = fr * 2^e, fr in [0.5, 1)
  double m = std::nearbyint((fr * 2.0 - 1.0) * 8.0);    // mantissa of a = (1 + m/8) 2^(e-1)
  int ex = e - 1;
  if (m == 8.0) {
    m = 0.0;
    ++ex;
  }
  const int code = ((ex + 7) << 3) | static_cast<int>(m);
  return sign | static_cast<uint8_t>(code > 0x7E ? 0x7E : code);
}

}  // namespace

extern "C" ess_status ess_compact_rows(const uint16_t* rows_bf16, int64_t n_rows, uint8_t* out) {
  if (n_rows < 0 || (n_rows > 0 && (!rows_bf16 || !out))) return ESS_ERR_INVALID_ARG;
  for (int64_t r = 0; r < n_rows; ++r) {
    const uint16_t* row = rows_bf16 + r * ess::kRowDim;
    uint8_t* dst = out + r * kCompactBytes;
    for (int j = 0; j < kTiles; ++j) {
      float amax = 0.0f;
      for (int i = 0; i < kTile; ++i) amax = std::fmax(amax, std::fabs(bf16_to_float(row[j * kTile + i])));
      float scale = 1.0f;
      if (amax > 0.0f) {
        int e;
        const float fr = std::frexp(amax / 448.0f, &e);   // q = fr * 2^e, fr in [0.5, 1)
        scale = std::ldexp(1.0f, fr == 0.5f ? e - 1 : e);
      }
      for (int i = 0; i < kTile; ++i) {
        const float q = bf16_to_float(row[j * kTile + i]) / scale;
        dst[j * kTile + i] = e4m3_encode(q);
      }
      std::memcpy(dst + ess::kLatent + 4 * j, &scale, 4);   // little-endian float32
    }
    std::memcpy(dst + ess::kLatent + 4 * kTiles, row + ess::kLatent,
                2 * (ess::kRowDim - ess::kLatent));
  }
  return ESS_OK;
}
