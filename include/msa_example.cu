// Calling libmsa from C++ without Python: builds q [1, 4, N, 128] and k, v
// [1, 2, N, 128] in device memory, runs vertical-slash attention on query
// heads 0 and 1, block-sparse on head 2 and streaming on head 3 into one
// output tensor, each call with its own workspace sized by the library; then
// the hierarchical pruning head on all four heads into a second output, and
// the workspace-free vertical-slash call into a third.  It checks the host
// status codes, the device status words and that every output value was
// written and is finite.  Exits 0 on success.
//
//   nvcc -std=c++17 -I include include/msa_example.cu \
//        -L dynamic_sparse_attention_slash_gb300 -l:libmsa.so \
//        -Xlinker -rpath=$PWD/dynamic_sparse_attention_slash_gb300 -o msa_example
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <vector>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "msa.h"

namespace {

msa_tensor view(void* p, int64_t B, int64_t H, int64_t N) {
  msa_tensor t;
  t.data = p;
  t.B = B;
  t.H = H;
  t.N = N;
  t.D = 128;
  t.sn = 128;  // contiguous [B][H][N][128]
  t.sh = N * 128;
  t.sb = H * N * 128;
  return t;
}

bool ok(int rc, const char* what) {
  if (rc != MSA_OK) std::fprintf(stderr, "%s: %s\n", what, msa_status_string(rc));
  return rc == MSA_OK;
}

}  // namespace

int main() {
  const int64_t B = 1, Hq = 4, Hkv = 2, N = 4096, D = 128;
  const size_t nq = B * Hq * N * D, nk = B * Hkv * N * D;
  // deterministic pseudo-random inputs in [-1, 1)
  uint32_t state = 12345u;
  auto rnd = [&state]() {
    state = state * 1664525u + 1013904223u;
    return static_cast<float>((state >> 8) & 0xffffu) / 32768.f - 1.f;
  };
  std::vector<__nv_bfloat16> hq(nq), hk(nk), hv(nk), hout(nq);
  for (auto& x : hq) x = __float2bfloat16(rnd());
  for (auto& x : hk) x = __float2bfloat16(rnd());
  for (auto& x : hv) x = __float2bfloat16(rnd());

  void *dq, *dk, *dv, *dout, *dout2, *dout3;
  if (cudaMalloc(&dq, nq * 2) || cudaMalloc(&dk, nk * 2) || cudaMalloc(&dv, nk * 2) ||
      cudaMalloc(&dout, nq * 2) || cudaMalloc(&dout2, nq * 2) || cudaMalloc(&dout3, nq * 2))
    return 1;
  cudaMemcpy(dq, hq.data(), nq * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dk, hk.data(), nk * 2, cudaMemcpyHostToDevice);
  cudaMemcpy(dv, hv.data(), nk * 2, cudaMemcpyHostToDevice);
  cudaMemset(dout, 0xff, nq * 2);  // NaN pattern: every value must be overwritten
  cudaMemset(dout2, 0xff, nq * 2);
  cudaMemset(dout3, 0xff, nq * 2);

  msa_tensor tq = view(dq, B, Hq, N), tk = view(dk, B, Hkv, N), tv = view(dv, B, Hkv, N),
             tout = view(dout, B, Hq, N);
  const int32_t vs_heads[2] = {0, 1}, bs_heads[1] = {2}, st_heads[1] = {3};
  const int64_t vertical_topk = 256, slash = 512, topk = 8, init_num = 1, local = 4;
  const size_t need[3] = {
      msa_workspace_bytes(MSA_KIND_VERTICAL_SLASH, &tq, &tk, vertical_topk, slash, 2),
      msa_workspace_bytes(MSA_KIND_BLOCK_SPARSE, &tq, &tk, topk, 0, 1),
      msa_workspace_bytes(MSA_KIND_STREAMING, &tq, &tk, init_num, local, 1)};
  void* ws[3];
  for (int i = 0; i < 3; ++i)
    if (need[i] == 0 || cudaMalloc(&ws[i], need[i])) return 1;  // cudaMalloc: 256-byte aligned

  msa_opts o = {};  // defaults: legacy stream, last_q 64, scale 1/sqrt(128)
  o.heads = vs_heads;
  o.n_heads = 2;
  o.workspace = ws[0];
  o.workspace_bytes = need[0];
  if (!ok(msa_vertical_slash(&tq, &tk, &tv, vertical_topk, slash, &tout, &o), "vertical-slash"))
    return 1;
  o.heads = bs_heads;
  o.n_heads = 1;
  o.workspace = ws[1];
  o.workspace_bytes = need[1];
  if (!ok(msa_block_sparse(&tq, &tk, &tv, topk, &tout, &o), "block-sparse")) return 1;
  o.heads = st_heads;
  o.workspace = ws[2];
  o.workspace_bytes = need[2];
  if (!ok(msa_streaming(&tq, &tk, &tv, init_num, local, &tout, &o), "streaming")) return 1;

  // hierarchical pruning on every head: chunks of 8, 2 and 1 blocks keeping 4, 6, 8
  msa_tensor tout2 = view(dout2, B, Hq, N);
  const msa_hip_stage stages[3] = {{8, 4}, {2, 6}, {1, 8}};
  const size_t need_hip = msa_workspace_bytes(MSA_KIND_HIERARCHICAL, &tq, &tk, 8, 0, 0);
  void* ws_hip;
  if (need_hip == 0 || cudaMalloc(&ws_hip, need_hip)) return 1;
  msa_opts oh = {};
  oh.workspace = ws_hip;
  oh.workspace_bytes = need_hip;
  if (!ok(msa_hierarchical(&tq, &tk, &tv, stages, 3, &tout2, &oh), "hierarchical")) return 1;
  // vertical-slash with the library's own scratch array (no workspace)
  msa_tensor tout3 = view(dout3, B, Hq, N);
  if (!ok(msa_vertical_slash_static(&tq, &tk, &tv, vertical_topk, slash, &tout3, nullptr),
          "vertical-slash (static scratch)"))
    return 1;

  for (int i = 0; i < 3; ++i)  // synchronises; a bounded wait that ran out would show here
    if (!ok(msa_device_status(ws[i], nullptr), "device status")) return 1;
  if (!ok(msa_device_status(ws_hip, nullptr), "device status (hierarchical)")) return 1;
  if (!ok(msa_vertical_slash_static_status(nullptr), "device status (static scratch)")) return 1;
  for (void* d : {dout, dout2, dout3}) {
    cudaMemcpy(hout.data(), d, nq * 2, cudaMemcpyDeviceToHost);
    for (size_t i = 0; i < nq; ++i)
      if (!std::isfinite(__bfloat162float(hout[i]))) {
        std::fprintf(stderr, "output value %zu not written\n", i);
        return 1;
      }
  }
  std::printf("msa_example ok: %lld kernel launches\n",
              static_cast<long long>(msa_kernel_launches()));
  return 0;
}
