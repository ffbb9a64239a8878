// Create-time repack of canonical affine-quantised weights into the GPU
// layout described in internal.h.  Host code, run once per handle.
#include <cstring>
#include <thread>
#include <vector>

#include "repack.h"

namespace moe {

// One canonical 4-bit row of K codes -> one qrow of qrow_bytes(K) bytes.
static void repack_row4(const uint8_t* q, const uint16_t* scale, const uint16_t* bias, int64_t K,
                        uint8_t* dst) {
  const int64_t words = K / 8;
  uint32_t* out = reinterpret_cast<uint32_t*>(dst);
  for (int64_t w = 0; w < words; ++w) {
    uint32_t orig;  // canonical: column 8w + c in nibble c (low nibble = even column)
    std::memcpy(&orig, q + 4 * w, 4);
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (orig >> (4 * i)) & 0xFu;        // column 8w + i
      const uint32_t hi = (orig >> (4 * (i + 4))) & 0xFu;  // column 8w + 4 + i
      v |= (lo | (hi << 4)) << (8 * i);
    }
    out[w] = v;
  }
  uint32_t* sb = reinterpret_cast<uint32_t*>(dst + K / 2);
  for (int64_t g = 0; g < K / kGroup; ++g)
    sb[g] = static_cast<uint32_t>(scale[g]) | (static_cast<uint32_t>(bias[g]) << 16);
  const int64_t used = K / 2 + K / kGroup * 4;
  std::memset(dst + used, 0, qrow_bytes(K) - used);
}

static void repack_rows(const moe_qtensor& t, int64_t row0, int64_t nrows, int64_t K,
                        uint8_t* dst, int64_t dst_stride) {
  for (int64_t r = row0; r < row0 + nrows; ++r)
    repack_row4(t.q + r * K / 2, t.scale + r * (K / kGroup), t.bias + r * (K / kGroup), K,
                dst + (r - row0) * dst_stride);
}

void repack_matrix(const moe_qtensor& t, int64_t rows, int64_t K, uint8_t* dst) {
  parallel_for(rows, [&](int64_t r) { repack_rows(t, r, 1, K, dst + r * qrow_bytes(K), qrow_bytes(K)); });
}

int64_t expert_blob_bytes(const Dims& d) {
  return d.I * 2 * qrow_bytes(d.D) + d.D * qrow_bytes(d.I);
}

void repack_expert(const Dims& d, const moe_qtensor& gate, const moe_qtensor& up,
                   const moe_qtensor& down, uint8_t* blob) {
  const int64_t rbD = qrow_bytes(d.D), rbI = qrow_bytes(d.I);
  for (int64_t j = 0; j < d.I; ++j) {
    repack_rows(gate, j, 1, d.D, blob + (2 * j) * rbD, rbD);
    repack_rows(up, j, 1, d.D, blob + (2 * j + 1) * rbD, rbD);
  }
  repack_rows(down, 0, d.D, d.I, blob + d.I * 2 * rbD, rbI);
}

int64_t layer_fixed_bytes(const Dims& d) {
  return router_t_bytes(d) + router_sb_bytes(d) + bias_bytes(d) + shared_gu_bytes(d) +
         shared_dn_bytes(d);
}

void repack_layer_fixed(const Dims& d, const moe_layer_weights& w, uint8_t* dst) {
  // router: [E][D] codes -> [D][E]; scale/bias [E][D/64] -> [D/64][E] words
  uint8_t* rt = dst;
  for (int64_t e = 0; e < d.E; ++e)
    for (int64_t c = 0; c < d.D; ++c) rt[c * d.E + e] = w.router.q[e * d.D + c];
  uint32_t* rsb = reinterpret_cast<uint32_t*>(dst + router_t_bytes(d));
  const int64_t ng = d.D / kGroup;
  for (int64_t e = 0; e < d.E; ++e)
    for (int64_t g = 0; g < ng; ++g)
      rsb[g * d.E + e] = static_cast<uint32_t>(w.router.scale[e * ng + g]) |
                         (static_cast<uint32_t>(w.router.bias[e * ng + g]) << 16);
  float* lb = reinterpret_cast<float*>(dst + router_t_bytes(d) + router_sb_bytes(d));
  std::memset(lb, 0, bias_bytes(d));
  for (int64_t e = 0; e < d.E; ++e) lb[e] = w.router_logit_bias ? w.router_logit_bias[e] : 0.f;
  uint8_t* gu = dst + router_t_bytes(d) + router_sb_bytes(d) + bias_bytes(d);
  const int64_t rbD = qrow_bytes(d.D), rbS = qrow_bytes(d.S);
  for (int64_t j = 0; j < d.S; ++j) {
    repack_rows(w.shared_gate, j, 1, d.D, gu + (2 * j) * rbD, rbD);
    repack_rows(w.shared_up, j, 1, d.D, gu + (2 * j + 1) * rbD, rbD);
  }
  uint8_t* dn = gu + shared_gu_bytes(d);
  repack_rows(w.shared_down, 0, d.D, d.S, dn, rbS);
}

void parallel_for(int64_t n, const std::function<void(int64_t)>& fn) {
  unsigned nt = std::thread::hardware_concurrency();
  if (nt == 0) nt = 4;
  if (nt > 32) nt = 32;
  if (n < static_cast<int64_t>(nt)) nt = static_cast<unsigned>(n);
  if (nt <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> th;
  th.reserve(nt);
  for (unsigned t = 0; t < nt; ++t)
    th.emplace_back([&, t] {
      for (int64_t i = t; i < n; i += nt) fn(i);
    });
  for (auto& x : th) x.join();
}

}  // namespace moe
