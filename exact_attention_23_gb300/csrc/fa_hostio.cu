// Attention forward over host-resident tensors (fa_fwd_host). The B·H heads are taken in
// chunks: each chunk's q, k, v are copied into a device staging buffer, attended by the
// fa_fwd kernel, and its o, lse copied back. Copies in, computation and copies out run on
// three streams with kSlots staging buffers, so the transfers of one chunk overlap the
// computation of its neighbours. Host-side orchestration only.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"
#include "fa_host.h"

namespace {

using fa::host::check_device;
using fa::host::overlaps;

constexpr int kMaxDev = 64;
constexpr size_t kAlign = 256;
// Staging buffers: with three, a chunk can be copied in while the previous one is attended
// and the one before it copied out.
constexpr int kSlots = 3;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// One staging buffer for c heads: q | k | v | o (bf16 [c][T][d]) | lse (fp32 [c][T]).
struct Chunk {
  size_t q, k, v, o, lse, bytes;
};
Chunk chunk_layout(long long c, long long T, long long d) {
  const size_t t = round_up(static_cast<size_t>(c * T * d * 2));
  Chunk L;
  L.q = 0;
  L.k = t;
  L.v = 2 * t;
  L.o = 3 * t;
  L.lse = 4 * t;
  L.bytes = 4 * t + round_up(static_cast<size_t>(c * T * 4));
  return L;
}

// Heads per chunk when the caller leaves it to the library: enough (head, pair of 128-row
// Q tiles) work units per launch to give every SM two, and no more heads than exist.
long long auto_heads(long long BH, long long T, int sms) {
  const long long pairs = (T + 255) / 256;
  const long long c = (2LL * sms + pairs - 1) / pairs;
  return std::max(1LL, std::min(c, BH));
}

bool sizes_ok(int B, int H, int T, int d) {
  if (B <= 0 || H <= 0 || T <= 0 || (d != 64 && d != 128)) return false;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > INT32_MAX) return false;
  if (static_cast<long long>(T) * d * 2 >= (1LL << 40)) return false;  // fa_fwd's TMA stride limit
  return BH * T * d < (1LL << 61) / 2;
}

// The copy streams of a device: created on first use and kept for the process (like the
// cached device properties, not per-call state).
struct CopyStreams {
  cudaStream_t in = nullptr, out = nullptr;
};
CopyStreams g_streams[kMaxDev];
std::once_flag g_streams_once[kMaxDev];

bool copy_streams(int dev, CopyStreams* s) {
  if (dev < 0 || dev >= kMaxDev) return false;
  std::call_once(g_streams_once[dev], [dev] {
    if (cudaStreamCreateWithFlags(&g_streams[dev].in, cudaStreamNonBlocking) != cudaSuccess)
      g_streams[dev].in = nullptr;
    if (cudaStreamCreateWithFlags(&g_streams[dev].out, cudaStreamNonBlocking) != cudaSuccess)
      g_streams[dev].out = nullptr;
  });
  *s = g_streams[dev];
  return s->in != nullptr && s->out != nullptr;
}

long long resolve_heads(long long BH, int T, int heads_per_chunk, bool* ok) {
  *ok = true;
  if (heads_per_chunk > 0) return std::min<long long>(heads_per_chunk, BH);
  int dev = -1, sms = 0;
  if (check_device(&dev, &sms) != FA_OK) {
    *ok = false;
    return 0;
  }
  return auto_heads(BH, T, sms);
}

}  // namespace

extern "C" {

size_t fa_fwd_host_workspace_size(int B, int H, int T, int d, int heads_per_chunk) {
  if (!sizes_ok(B, H, T, d) || heads_per_chunk < 0) return 0;
  bool ok = false;
  const long long c = resolve_heads(static_cast<long long>(B) * H, T, heads_per_chunk, &ok);
  if (!ok) return 0;
  return kSlots * chunk_layout(c, T, d).bytes;
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int T, int d, int causal, float scale, int heads_per_chunk, void* workspace,
                size_t workspace_bytes, void* stream) {
  // ---- host-side validation: nothing is enqueued on failure
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (!sizes_ok(B, H, T, d) || heads_per_chunk < 0) return FA_ERR_INVALID_ARG;
  if (!fa::host::scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return FA_ERR_MISALIGNED;
  const long long BH = static_cast<long long>(B) * H;
  const size_t tbytes = static_cast<size_t>(BH * T * d * 2);
  const size_t lbytes = static_cast<size_t>(BH * T * 4);
  if (overlaps(o, tbytes, q, tbytes) || overlaps(o, tbytes, k, tbytes) ||
      overlaps(o, tbytes, v, tbytes) || overlaps(lse, lbytes, q, tbytes) ||
      overlaps(lse, lbytes, k, tbytes) || overlaps(lse, lbytes, v, tbytes) ||
      overlaps(lse, lbytes, o, tbytes))
    return FA_ERR_INVALID_ARG;
  bool ok = false;
  const long long c = resolve_heads(BH, T, heads_per_chunk, &ok);
  if (!ok) return FA_ERR_UNSUPPORTED_DEVICE;
  const Chunk L = chunk_layout(c, T, d);
  if (workspace_bytes < kSlots * L.bytes) return FA_ERR_INVALID_ARG;

  int dev = -1, sms = 0;
  const int dst = check_device(&dev, &sms);
  if (dst != FA_OK) return dst;
  CopyStreams cs;
  if (!copy_streams(dev, &cs)) return FA_ERR_LAUNCH;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);

  // ev_start: work already on `stream` (an earlier call using this workspace ends there);
  // ev_in[s] / ev_done[s] / ev_out[s]: the latest chunk in slot s copied in / attended /
  // copied out.
  cudaEvent_t ev_start = nullptr, ev_in[kSlots] = {}, ev_done[kSlots] = {}, ev_out[kSlots] = {};
  cudaEvent_t* all[1 + 3 * kSlots];
  all[0] = &ev_start;
  for (int s = 0; s < kSlots; ++s) {
    all[1 + s] = &ev_in[s];
    all[1 + kSlots + s] = &ev_done[s];
    all[1 + 2 * kSlots + s] = &ev_out[s];
  }
  int rc = FA_OK;
  for (cudaEvent_t* e : all)
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) rc = FA_ERR_LAUNCH;

  auto cu = [&](cudaError_t e) {
    if (e != cudaSuccess && rc == FA_OK) rc = FA_ERR_LAUNCH;
    return rc == FA_OK;
  };
  const auto* qh = static_cast<const uint8_t*>(q);
  const auto* kh = static_cast<const uint8_t*>(k);
  const auto* vh = static_cast<const uint8_t*>(v);
  auto* oh = static_cast<uint8_t*>(o);
  auto* lh = reinterpret_cast<uint8_t*>(lse);
  auto* ws = static_cast<uint8_t*>(workspace);
  const size_t head_t = static_cast<size_t>(T) * d * 2;  // bytes of one head of q/k/v/o
  const size_t head_l = static_cast<size_t>(T) * 4;      // bytes of one head of lse
  const long long n_chunks = (BH + c - 1) / c;
  long long last = -1;

  if (rc == FA_OK && cu(cudaEventRecord(ev_start, st)) && cu(cudaStreamWaitEvent(cs.in, ev_start, 0))) {
    for (long long i = 0; i < n_chunks && rc == FA_OK; ++i) {
      const int s = static_cast<int>(i % kSlots);
      const long long h0 = i * c;
      const int hc = static_cast<int>(std::min(c, BH - h0));
      uint8_t* buf = ws + s * L.bytes;
      // The slot's previous chunk must have been copied out before its buffer is refilled.
      if (i >= kSlots && !cu(cudaStreamWaitEvent(cs.in, ev_out[s], 0))) break;
      const size_t nb = hc * head_t;
      if (!cu(cudaMemcpyAsync(buf + L.q, qh + h0 * head_t, nb, cudaMemcpyHostToDevice, cs.in)) ||
          !cu(cudaMemcpyAsync(buf + L.k, kh + h0 * head_t, nb, cudaMemcpyHostToDevice, cs.in)) ||
          !cu(cudaMemcpyAsync(buf + L.v, vh + h0 * head_t, nb, cudaMemcpyHostToDevice, cs.in)) ||
          !cu(cudaEventRecord(ev_in[s], cs.in)) || !cu(cudaStreamWaitEvent(st, ev_in[s], 0)))
        break;
      const int frc = fa_fwd(buf + L.q, buf + L.k, buf + L.v, buf + L.o,
                             reinterpret_cast<float*>(buf + L.lse), 1, hc, T, d, causal, scale,
                             stream);
      if (frc != FA_OK) {
        rc = frc;
        break;
      }
      if (!cu(cudaEventRecord(ev_done[s], st)) || !cu(cudaStreamWaitEvent(cs.out, ev_done[s], 0)) ||
          !cu(cudaMemcpyAsync(oh + h0 * head_t, buf + L.o, nb, cudaMemcpyDeviceToHost, cs.out)) ||
          !cu(cudaMemcpyAsync(lh + h0 * head_l, buf + L.lse, hc * head_l, cudaMemcpyDeviceToHost,
                              cs.out)) ||
          !cu(cudaEventRecord(ev_out[s], cs.out)))
        break;
      last = i;
    }
  }
  // `stream` waits for the last copy out (the copy-out stream runs in order), so that
  // synchronising it makes o and lse readable and a later call may reuse the workspace;
  // and for every copy in (after an error a chunk may have been copied in but not attended).
  if (last >= 0) cudaStreamWaitEvent(st, ev_out[last % kSlots], 0);
  if (ev_start && cudaEventRecord(ev_start, cs.in) == cudaSuccess)
    cudaStreamWaitEvent(st, ev_start, 0);
  for (cudaEvent_t* e : all)
    if (*e) cudaEventDestroy(*e);  // released once pending work completes
  return rc;
}

}  // extern "C"
