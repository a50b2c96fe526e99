// stream_floor.cu -- the streaming floor of one GB300: how fast a kernel that only moves bytes
// can read a contiguous region of HBM into shared memory, one CTA per SM, the way the decode
// kernels stage their K/V (a ring of shared-memory stages filled by cp.async.bulk copies and
// released by consumer warps that compute nothing).  It bounds what a decode-attention launch
// of a given size can reach: a cold single launch of one layer's 16K-token prefix (67 MB) pays
// its ramp and tail, which a 1 GB launch amortises; a chain of back-to-back launches with
// programmatic dependent launch (each waits on the previous one, as the decode kernels do)
// shows the per-launch floor inside a model step.
//
// Every wait is bounded (1 s); on expiry the kernel sets an error word the host reads and
// stops.  A measurement tool, not part of the library: built and run by stream_floor.py.
//
//   stream_floor [peak_GBps]      prints one line per case: bytes, us, GB/s, fraction of peak
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

namespace {

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(uint32_t a, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_expect(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ bool bar_test(uint32_t a, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(a), "r"(parity)
      : "memory");
  return done != 0;
}
// true once the phase with this parity has completed; false (and the error word set) after 1 s
__device__ __forceinline__ bool bar_wait(uint32_t a, uint32_t parity, int* err) {
  const uint64_t t0 = now_ns();
  while (!bar_test(a, parity))
    if (now_ns() - t0 > 1000000000ull) {
      atomicExch(err, 1);
      return false;
    }
  return true;
}
__device__ __forceinline__ void copy_in(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// CTA i streams bytes [i * window, (i + 1) * window) of src through n_stages stages of
// stage_bytes, each filled by stage_bytes / copy_bytes bulk copies (issued by the producer
// warp's lanes); the consumer warp waits for each stage, touches one word of it and releases it.
// window is a multiple of stage_bytes, copy_bytes divides stage_bytes, both multiples of 16.
__global__ void __launch_bounds__(64, 1)
    stream_kernel(const char* src, int64_t window, int stage_bytes, int n_stages, int copy_bytes, int* err,
                  float* sink) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t bars = base + (uint32_t)(n_stages * stage_bytes);
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (n_stages + s); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < n_stages; ++s) {
      bar_init(full(s), 1);
      bar_init(empty(s), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // as the decode kernels do: read only after the previous kernel in the stream has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const char* mine = src + (int64_t)blockIdx.x * window;
  const int n_fill = (int)(window / stage_bytes);
  const int copies = stage_bytes / copy_bytes;
  if (warp == 0) {
    int n = 0;
    for (; n < n_fill; ++n) {
      const int s = n % n_stages;
      const bool free_ok = n < n_stages || bar_wait(empty(s), ((n / n_stages) - 1) & 1, err);
      if (!__all_sync(0xffffffffu, free_ok)) break;
      if (lane == 0) bar_expect(full(s), (uint32_t)stage_bytes);
      __syncwarp();
      for (int c = lane; c < copies; c += 32)
        copy_in(base + (uint32_t)(s * stage_bytes + c * copy_bytes), mine + (int64_t)n * stage_bytes + (int64_t)c * copy_bytes,
                (uint32_t)copy_bytes, full(s));
    }
    // leave with no copy in flight
    if (lane == 0)
      for (int i = max(0, n - n_stages); i < n; ++i) bar_wait(full(i % n_stages), (i / n_stages) & 1, err);
  } else {
    float acc = 0.f;
    for (int n = 0; n < n_fill; ++n) {
      const int s = n % n_stages;
      const bool ok = bar_wait(full(s), (n / n_stages) & 1, err);
      if (!__all_sync(0xffffffffu, ok)) break;
      acc += reinterpret_cast<const float*>(smem + (size_t)s * stage_bytes)[lane];
      __syncwarp();
      if (lane == 0) bar_arrive(empty(s));
    }
    if (acc == 1234.5f) sink[0] = acc;  // keeps the loads
  }
}

cudaError_t launch(const char* src, int grid, int smem, int64_t window, int stage, int n_stages, int copy, int* err,
                   float* sink, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(64);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stream_kernel, src, window, stage, n_stages, copy, err, sink);
}

#define CHECK(x)                                                                        \
  do {                                                                                  \
    cudaError_t e_ = (x);                                                               \
    if (e_ != cudaSuccess) {                                                            \
      std::fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));              \
      std::exit(2);                                                                     \
    }                                                                                   \
  } while (0)

}  // namespace

int main(int argc, char** argv) {
  const double peak = argc > 1 ? std::atof(argv[1]) : 0.0;
  int n_sm = 0;
  CHECK(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, 0));
  const int64_t total = 4LL << 30;  // 4 GiB of regions to read, L2 (129 MB) many times over
  char* buf = nullptr;
  int* err = nullptr;
  float* sink = nullptr;
  CHECK(cudaMalloc(&buf, total));
  CHECK(cudaMemset(buf, 1, total));
  CHECK(cudaMalloc(&err, sizeof(int)));
  CHECK(cudaMemset(err, 0, sizeof(int)));
  CHECK(cudaMalloc(&sink, sizeof(float)));
  CHECK(cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024));
  char* flush = nullptr;  // written between single launches so that none finds its bytes in L2
  const size_t flush_bytes = 256u << 20;
  CHECK(cudaMalloc(&flush, flush_bytes));
  cudaStream_t st;
  CHECK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  cudaEvent_t e0, e1;
  CHECK(cudaEventCreate(&e0));
  CHECK(cudaEventCreate(&e1));

  struct Ring {
    int stage, n_stages, copy;
    const char* name;
  };
  const Ring rings[] = {
      {65536, 3, 2048, "3 x 64 KB stages, 2 KB copies"},   // the decode kernels' ring and row copies
      {65536, 3, 32768, "3 x 64 KB stages, 32 KB copies"},
  };
  std::printf("# %d SMs, one CTA per SM; peak %.1f GB/s\n", n_sm, peak);
  for (const Ring& r : rings) {
    const int smem = r.stage * r.n_stages + 16 * r.n_stages + 64;
    for (const int64_t per_launch : {67108864LL, 1073741824LL}) {
      const int64_t window = per_launch / n_sm / r.stage * r.stage;
      const int64_t bytes = window * n_sm;
      const int regions = (int)(total / bytes);
      // single cold launches: L2 flushed before each, median of 9 after 2 untimed
      std::vector<float> t;
      for (int rep = 0; rep < 11; ++rep) {
        CHECK(cudaMemsetAsync(flush, rep & 0xff, flush_bytes, st));
        CHECK(cudaEventRecord(e0, st));
        CHECK(launch(buf + (int64_t)(rep % regions) * bytes, n_sm, smem, window, r.stage, r.n_stages, r.copy, err,
                     sink, st));
        CHECK(cudaEventRecord(e1, st));
        CHECK(cudaEventSynchronize(e1));
        float ms = 0.f;
        CHECK(cudaEventElapsedTime(&ms, e0, e1));
        if (rep >= 2) t.push_back(ms);
      }
      std::sort(t.begin(), t.end());
      const double us = 1e3 * t[t.size() / 2];
      const double gbs = bytes / (us * 1e-6) / 1e9;
      std::printf("single launch | %-31s | %7.1f MB | %8.2f us | %6.0f GB/s | %.3f of peak\n", r.name, bytes / 1e6,
                  us, gbs, peak > 0 ? gbs / peak : 0.0);
      if (per_launch > 67108864LL) continue;
      // a chain of back-to-back launches on distinct regions (a model step's layers)
      const int chain = std::min(regions, 32);
      std::vector<float> c;
      for (int rep = 0; rep < 7; ++rep) {
        CHECK(cudaMemsetAsync(flush, rep & 0xff, flush_bytes, st));
        CHECK(cudaEventRecord(e0, st));
        for (int k = 0; k < chain; ++k)
          CHECK(launch(buf + (int64_t)k * bytes, n_sm, smem, window, r.stage, r.n_stages, r.copy, err, sink, st));
        CHECK(cudaEventRecord(e1, st));
        CHECK(cudaEventSynchronize(e1));
        float ms = 0.f;
        CHECK(cudaEventElapsedTime(&ms, e0, e1));
        if (rep >= 2) c.push_back(ms);
      }
      std::sort(c.begin(), c.end());
      const double us_each = 1e3 * c[c.size() / 2] / chain;
      const double gbs_c = bytes / (us_each * 1e-6) / 1e9;
      std::printf("chain of %2d    | %-31s | %7.1f MB | %8.2f us | %6.0f GB/s | %.3f of peak (per launch)\n", chain,
                  r.name, bytes / 1e6, us_each, gbs_c, peak > 0 ? gbs_c / peak : 0.0);
    }
  }
  int h_err = 0;
  CHECK(cudaMemcpy(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost));
  if (h_err) {
    std::fprintf(stderr, "a bounded wait gave up\n");
    return 3;
  }
  return 0;
}
