// Host-side checks run under AddressSanitizer and UndefinedBehaviorSanitizer
// (built and run by test_sanitizers.py, no GPU needed).
//
// Part 1 exercises the FP64 oracle's entry points on small problems with the
// edge cases they must handle (empty contexts, partial pages, empty splits,
// row selection, FP8 caches, padding and out-of-range ids) and checks that
// they agree with one another. Part 2 drives the library's C ABI through
// every argument check that runs before a CUDA call, plus the host-only
// planner, so the host code of the library is exercised under the
// sanitizers too. Any sanitizer report aborts the program; a failed check
// returns 1.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <random>
#include <vector>

#include "paged_decode_attn.h"

extern "C" {
void oracle_round_array(const double* x, int64_t n, int dtype, uint16_t* bits_out,
                        double* rounded_out);
int oracle_paged_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                        const int32_t* block_table, const int32_t* context_lens, int B, int Hq,
                        int Hkv, int D, int block_size, int max_blocks, int64_t num_blocks,
                        int dtype, double scale, double* out, int num_threads);
int oracle_paged_decode_rows(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                             const int32_t* block_table, const int32_t* context_lens, int B,
                             int Hq, int Hkv, int D, int block_size, int max_blocks,
                             int64_t num_blocks, int dtype, double scale, const int32_t* rows,
                             int64_t n_rows, double* out_rows, int num_threads);
int oracle_paged_decode_kv(const uint16_t* q, const void* k_cache, const void* v_cache,
                           int kv_dtype, const double* k_scale, const double* v_scale,
                           const int32_t* block_table, const int32_t* context_lens, int B,
                           int Hq, int Hkv, int D, int block_size, int max_blocks,
                           int64_t num_blocks, int q_dtype, double scale, const int32_t* rows,
                           int64_t n_rows, double* out_rows, int num_threads);
int oracle_split_partials(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                          const int32_t* block_table, const int32_t* context_lens, int B, int Hq,
                          int Hkv, int D, int block_size, int max_blocks, int64_t num_blocks,
                          int dtype, double scale, int chunk_pages, int num_splits,
                          double* lse, double* o);
int oracle_lse_merge(const double* lse, const double* o, int64_t n_rows, int num_splits, int D,
                     double* out);
int oracle_rope_kv_write(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* positions, const int64_t* slot_mapping,
                         const float* cos_sin, int T, int Hq, int Hkv, int D, int rot_dim,
                         int max_position, int neox, int64_t num_slots, int dtype,
                         uint16_t* q_out, uint16_t* k_cache, uint16_t* v_cache);
int oracle_copy_blocks(uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                       int64_t block_bytes, const int64_t* pairs, int64_t n_pairs);
int oracle_gather_kv(const uint8_t* k_cache, const uint8_t* v_cache, int64_t num_blocks,
                     int block_size, int64_t row_bytes, const int32_t* block_table,
                     int max_blocks, const int32_t* lens, int B, uint8_t* k_out,
                     uint8_t* v_out);
int oracle_scatter_kv(const uint8_t* k_in, const uint8_t* v_in, int64_t n_rows,
                      int64_t row_bytes, const int64_t* slot_mapping, uint8_t* k_cache,
                      uint8_t* v_cache, int64_t num_slots);
int oracle_remap_table(int32_t* block_table, int B, int max_blocks, const int32_t* lens,
                       int block_size, const int32_t* new_id, int64_t num_blocks);
}

namespace {

int g_failures = 0;

void expect(bool ok, const char* what) {
  if (!ok) {
    std::fprintf(stderr, "FAILED: %s\n", what);
    ++g_failures;
  }
}

std::vector<uint16_t> random_bf16(size_t n, std::mt19937& rng) {
  std::normal_distribution<double> nd(0.0, 1.0);
  std::vector<double> x(n);
  for (auto& v : x) v = nd(rng);
  std::vector<uint16_t> bits(n);
  oracle_round_array(x.data(), (int64_t)n, 0, bits.data(), nullptr);
  return bits;
}

void oracle_checks() {
  std::mt19937 rng(7);
  const int B = 3, Hq = 8, Hkv = 2, D = 16, bs = 4, max_blocks = 5, nb = 16;
  const int lens[B] = {0, 5, 13};
  auto q = random_bf16((size_t)B * Hq * D, rng);
  auto k = random_bf16((size_t)nb * bs * Hkv * D, rng);
  auto v = random_bf16((size_t)nb * bs * Hkv * D, rng);
  std::vector<int32_t> table((size_t)B * max_blocks);
  for (size_t i = 0; i < table.size(); ++i) table[i] = (int32_t)((i * 7 + 3) % nb);
  const double scale = 0.25;
  std::vector<double> full((size_t)B * Hq * D);
  expect(oracle_paged_decode(q.data(), k.data(), v.data(), table.data(), lens, B, Hq, Hkv, D, bs,
                             max_blocks, nb, 0, scale, full.data(), 3) == 0,
         "paged_decode");
  for (int d = 0; d < Hq * D; ++d) expect(full[d] == 0.0, "empty context gives zeros");

  std::vector<int32_t> rows = {2, 7, 1, 0, 2, 7, 0, 3};
  std::vector<double> sel(rows.size() / 2 * D);
  expect(oracle_paged_decode_rows(q.data(), k.data(), v.data(), table.data(), lens, B, Hq, Hkv,
                                  D, bs, max_blocks, nb, 0, scale, rows.data(),
                                  (int64_t)rows.size() / 2, sel.data(), 2) == 0,
         "paged_decode_rows");
  for (size_t r = 0; r < rows.size() / 2; ++r)
    for (int d = 0; d < D; ++d)
      expect(sel[r * D + d] == full[((size_t)rows[2 * r] * Hq + rows[2 * r + 1]) * D + d],
             "selected rows equal the full output");
  int32_t bad_rows[2] = {B, 0};
  expect(oracle_paged_decode_rows(q.data(), k.data(), v.data(), table.data(), lens, B, Hq, Hkv,
                                  D, bs, max_blocks, nb, 0, scale, bad_rows, 1, sel.data(),
                                  1) != 0,
         "a row outside the batch is rejected");

  for (int S = 1; S <= 5; ++S) {
    const int chunk = (max_blocks + S - 1) / S;
    std::vector<double> lse((size_t)B * Hq * S), o((size_t)B * Hq * S * D), merged(full.size());
    expect(oracle_split_partials(q.data(), k.data(), v.data(), table.data(), lens, B, Hq, Hkv, D,
                                 bs, max_blocks, nb, 0, scale, chunk, S, lse.data(),
                                 o.data()) == 0,
           "split_partials");
    expect(oracle_lse_merge(lse.data(), o.data(), (int64_t)B * Hq, S, D, merged.data()) == 0,
           "lse_merge");
    for (size_t i = 0; i < full.size(); ++i)
      expect(std::fabs(merged[i] - full[i]) < 1e-12, "split merge equals the unsplit result");
  }

  // FP8 caches with per-head scales (NaN codes avoided)
  std::vector<uint8_t> k8(k.size()), v8(v.size());
  for (size_t i = 0; i < k8.size(); ++i) {
    k8[i] = (uint8_t)(rng() % 0x7f) | (uint8_t)((rng() & 1) << 7);
    v8[i] = (uint8_t)(rng() % 0x7f) | (uint8_t)((rng() & 1) << 7);
  }
  const double ks[Hkv] = {0.5, 2.0}, vs[Hkv] = {0.125, 3.0};
  std::vector<double> out8(full.size());
  expect(oracle_paged_decode_kv(q.data(), k8.data(), v8.data(), 2, ks, vs, table.data(), lens, B,
                                Hq, Hkv, D, bs, max_blocks, nb, 0, scale, nullptr, 0,
                                out8.data(), 2) == 0,
         "paged_decode_kv fp8");
  for (double x : out8) expect(std::isfinite(x), "fp8 output finite");

  // RoPE + cache write: a padding slot, a position outside the table, a slot past the cache
  const int T = 4, rot = 8, max_pos = 6;
  auto qr = random_bf16((size_t)T * Hq * D, rng);
  auto kr = random_bf16((size_t)T * Hkv * D, rng);
  auto vr = random_bf16((size_t)T * Hkv * D, rng);
  std::vector<float> cs((size_t)max_pos * rot);
  for (size_t i = 0; i < cs.size(); ++i) cs[i] = (float)std::cos(0.1 * (double)i);
  const int32_t pos[T] = {0, 5, 9, 2};
  const int64_t slots[T] = {3, -1, 4, (int64_t)nb * bs};
  std::vector<uint16_t> qo(qr.size()), kc(k), vc(v);
  expect(oracle_rope_kv_write(qr.data(), kr.data(), vr.data(), pos, slots, cs.data(), T, Hq, Hkv,
                              D, rot, max_pos, 1, (int64_t)nb * bs, 0, qo.data(), kc.data(),
                              vc.data()) == 0,
         "rope_kv_write");

  // KV movement: scatter rows into slots, gather them back, copy and remap
  const int64_t row_bytes = (int64_t)Hkv * D * 2;
  std::vector<int64_t> smap = {5, 9, -1, 30};
  std::vector<uint8_t> kin((size_t)smap.size() * row_bytes), vin(kin.size());
  for (size_t i = 0; i < kin.size(); ++i) {
    kin[i] = (uint8_t)rng();
    vin[i] = (uint8_t)rng();
  }
  std::vector<uint8_t> kb(k.size() * 2), vb(v.size() * 2);
  expect(oracle_scatter_kv(kin.data(), vin.data(), (int64_t)smap.size(), row_bytes, smap.data(),
                           kb.data(), vb.data(), (int64_t)nb * bs) == 0,
         "scatter_kv");
  std::vector<uint8_t> kg((size_t)(lens[0] + lens[1] + lens[2]) * row_bytes), vg(kg.size());
  expect(oracle_gather_kv(kb.data(), vb.data(), nb, bs, row_bytes, table.data(), max_blocks, lens,
                          B, kg.data(), vg.data()) == 0,
         "gather_kv");
  const int64_t pairs[4] = {1, 14, 2, 15};
  expect(oracle_copy_blocks(kb.data(), vb.data(), nb, (int64_t)bs * row_bytes, pairs, 2) == 0,
         "copy_blocks");
  std::vector<int32_t> new_id(nb);
  for (int i = 0; i < nb; ++i) new_id[i] = (i * 5 + 1) % nb;
  std::vector<int32_t> t2(table);
  expect(oracle_remap_table(t2.data(), B, max_blocks, lens, bs, new_id.data(), nb) == 0,
         "remap_table");
}

void abi_checks() {
  expect(paged_decode_attn_abi_version() == PDA_ABI_VERSION, "abi version");
  pda_config c = {32, 8, 128, 16, PDA_BF16, 4, 2048, 64, 0, 0};
  int S = 0, chunk = 0;
  for (int sms : {1, 8, 148, 152})
    for (int b : {1, 4, 4})
      for (int mb : {1, 2, 513, 2048}) {
        expect(paged_decode_attn_plan(&c, sms, b, mb, 0, &S, &chunk) == PDA_OK, "plan");
        expect(S >= 1 && S <= 64 && chunk >= 1 && (int64_t)S * chunk >= mb, "plan covers pages");
      }
  expect(paged_decode_attn_plan(&c, 0, 1, 1, 0, &S, &chunk) == PDA_EINVAL, "plan num_sms 0");
  expect(paged_decode_attn_plan(nullptr, 1, 1, 1, 0, &S, &chunk) != PDA_OK, "plan null config");
  pda_handle h = nullptr;
  pda_config bad = c;
  bad.num_q_heads = 30;
  expect(paged_decode_attn_create(&bad, &h) == PDA_EINVAL && h == nullptr, "create Hq % Hkv");
  bad = c;
  bad.head_dim = 96;
  expect(paged_decode_attn_create(&bad, &h) == PDA_EUNSUPPORTED, "create head_dim 96");
  bad = c;
  bad.num_q_heads = 17 * bad.num_kv_heads;
  expect(paged_decode_attn_create(&bad, &h) == PDA_EUNSUPPORTED, "create group size 17");
  bad = c;
  bad.kv_fp8 = 1;
  bad.head_dim = 256;
  expect(paged_decode_attn_create(&bad, &h) == PDA_EUNSUPPORTED, "create fp8 head_dim 256");
  expect(std::strlen(paged_decode_attn_last_error()) > 0, "last_error set");
  expect(paged_decode_attn_create(nullptr, &h) != PDA_OK, "create null config");
  paged_decode_attn_destroy(nullptr);
  int x = 0, y = 0, z = 0, w = 0;
  expect(paged_decode_attn_run(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 1, 1, 1,
                               1.f, nullptr, nullptr) == PDA_EINVAL,
         "run null handle");
  expect(paged_decode_attn_launch_shape(nullptr, 1, 1, 0, 0, &x, &y, &z, &w) == PDA_EINVAL,
         "launch_shape null handle");
  expect(paged_decode_attn_check_device_error(nullptr, &x, &y, nullptr) == PDA_EINVAL,
         "check_device_error null handle");
  expect(paged_decode_attn_merge(nullptr, nullptr, 4, 65, 128, nullptr, PDA_F32, 0, nullptr) ==
             PDA_EINVAL,
         "merge num_splits 65");
  expect(paged_decode_attn_merge(nullptr, nullptr, 0, 4, 128, nullptr, PDA_F32, 0, nullptr) ==
             PDA_OK,
         "merge of no rows is a no-op");
  expect(paged_decode_attn_run_noalloc(nullptr, nullptr, nullptr, nullptr, nullptr, -1, 32, 8,
                                       128, 16, PDA_BF16, 1, 1, 1.f, nullptr, 0, 0,
                                       nullptr) == PDA_EINVAL,
         "noalloc negative batch");
  expect(paged_decode_attn_run_noalloc(nullptr, nullptr, nullptr, nullptr, nullptr, 0, 32, 8, 128,
                                       16, PDA_BF16, 1, 1, 1.f, nullptr, 0, 0,
                                       nullptr) == PDA_OK,
         "noalloc batch 0 is a no-op");
  expect(paged_decode_attn_copy_blocks(nullptr, nullptr, 1, 16, nullptr, 70000, nullptr, 0,
                                       nullptr) == PDA_EINVAL,
         "copy_blocks too many pairs");
  expect(paged_decode_attn_rope_kv_write(nullptr, 0, nullptr, 0, nullptr, 0, nullptr, nullptr,
                                         nullptr, 1, 8, 1, 1, 8, 8, 100, PDA_BF16, nullptr, 0,
                                         nullptr, nullptr, 1, nullptr, 0, nullptr) != PDA_OK,
         "rope_kv_write bad head_dim");
  // a valid configuration: a handle on a GPU host, a CUDA error (no driver) on a CPU host
  const int st = paged_decode_attn_create(&c, &h);
  expect(st == PDA_OK || st == PDA_ECUDA, "create with a valid configuration");
  if (st == PDA_OK) {
    expect(paged_decode_attn_launch_shape(h, 4, 2048, 0, 0, &x, &y, &z, &w) == PDA_OK,
           "launch_shape");
    paged_decode_attn_destroy(h);
  }
}

}  // namespace

int main() {
  oracle_checks();
  abi_checks();
  std::printf("sanitize_driver: %d failure(s)\n", g_failures);
  return g_failures == 0 ? 0 : 1;
}
