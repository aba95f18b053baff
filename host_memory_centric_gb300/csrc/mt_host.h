// mt_host.h -- host-side pieces of libmt that need no GPU: flat layout,
// seeded initialisation, BF16 rounding, Adam, the worker pool and the static
// prefetch schedule.  Internal header.
#pragma once
#include <stdint.h>

#include <atomic>
#include <condition_variable>
#include <deque>
#include <functional>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "../../include/mt.h"

namespace mth {

// ---------------------------------------------------------------- layout
// One block per layer ([Hotdry] layer-contiguous tiling; [Review] 3-2 (4)):
// regions W (bf16) | G (bf16) | master | m | v (fp32), each at a 4096-byte
// boundary of the block; the same tensors at the same element offsets in every
// region, each tensor starting on a multiple of 128 elements.
struct TensorDesc {
  int64_t off, rows, cols;
};
struct BlockDesc {
  TensorDesc t[MT_MAX_TENSORS];
  int nt = 0;
  int64_t n_real = 0, n_pad = 0;
  int64_t region[5] = {0, 0, 0, 0, 0};  // byte offsets of W, G, master, m, v
  int64_t wbytes = 0;                   // bytes of the W region (= G region)
  int64_t fbytes = 0;                   // bytes of one fp32 region
  int64_t bytes = 0, store_off = 0;
};
bool config_valid(const mt_config* c, std::string* why);
std::vector<BlockDesc> build_layout(const mt_config* c);
int64_t tokens_per_step(const mt_config* c);

// ---------------------------------------------------------------- numerics
uint16_t bf16_rne(float f);
float bf16_val(uint16_t b);
// Master values (n_pad floats) of block j: N(0, init_std) matrices from the
// block/tensor stream of SplitMix64, RMSNorm gains 1, padding 0.
void init_block(const mt_config* c, const BlockDesc& b, int j, float* master, int64_t e0, int64_t e1);
// Adam over [0, n) (FP32 arithmetic) on gradient g (BF16); when gcopy is not
// null the gradient is also written there (the slab unpack into the store's G
// region, fused into the same pass).  g == nullptr: a zero gradient (the
// experts of an MoE layer that no token was routed to).
void adam(int64_t n, const uint16_t* g, uint16_t* gcopy, float* th, float* m, float* v, uint16_t* w, int32_t t,
          float lr, float b1, float b2, float eps, float wd);
// Host gradient accumulation over micro-batch passes: acc = float(g) on the
// first pass, acc += float(g) on the later ones.
void accumulate(int64_t n, const uint16_t* g, float* acc, bool first);
// The last pass: the FP32 gradient acc + float(g) goes back into acc, as BF16
// into gcopy when not null, and drives the same Adam update.
void adam_acc(int64_t n, const uint16_t* g, float* acc, uint16_t* gcopy, float* th, float* m, float* v, uint16_t* w,
              int32_t t, float lr, float b1, float b2, float eps, float wd);
// Tokens one pass over the layers processes, and passes per step: with host
// accumulation every micro-batch is its own pass.
int64_t tokens_per_pass(const mt_config* c);
int passes_per_step(const mt_config* c);

// ---------------------------------------------------------------- worker pool
// Fixed threads running index ranges.  parallel_for may be called from several
// threads at once; the caller works on queued ranges while it waits.
class Pool {
 public:
  ~Pool() { stop(); }
  void start(int n);
  void stop();
  int size() const { return (int)threads_.size(); }
  // fn(i) for i in [0, n); returns false if any call threw (message in *err).
  // urgent: the n tasks go ahead of every queued task (in order), so a worker
  // takes them as soon as it finishes the task it is running.
  bool parallel_for(int64_t n, const std::function<void(int64_t)>& fn, std::string* err, bool urgent = false);

 private:
  // Completion count of one parallel_for, on the caller's stack.  Every
  // access after the tasks are queued happens under mu, so the caller, which
  // sees left == 0 only under mu, returns (and destroys the latch) only after
  // the last worker has released it.
  struct Latch {
    int64_t left = 0;
    std::mutex mu;
    std::condition_variable cv;
    bool bad = false;
    std::string msg;
  };
  struct Task {
    const std::function<void(int64_t)>* fn;
    int64_t i;
    Latch* latch;
  };
  bool run_own(const Latch* latch);
  void run(Task& t);
  std::vector<std::thread> threads_;
  std::mutex mu_;
  std::condition_variable cv_;
  std::deque<Task> q_;
  bool stop_ = false;
};

// ---------------------------------------------------------------- schedule
int32_t schedule(int32_t n, const double* b, const double* d, const double* c, const double* a, double bw_h2d,
                 double bw_d2h, double* stall);

// Steady-state model of the whole pipeline ([Peter] 記憶體預取策略: prefetch
// timed from each layer's bytes, the link bandwidth and its compute time),
// extended with the host side: the just-in-time pack, the K gradient slabs
// and host Adam.  One entry per visit of a step (the visit plan's order).
struct SimIn {
  int32_t n = 0;                   // visits per step
  const int32_t* kind = nullptr;   // 0 forward, 1 head, 2 recompute, 3 backward
  const int32_t* block = nullptr;  // block of the visit
  const double* b = nullptr;       // bytes copied host-to-device before the visit computes
  const double* p = nullptr;       // bytes packed on the host first (0 with a pinned store)
  const double* d = nullptr;       // gradient bytes exported after it (0: no export)
  const double* c = nullptr;       // compute seconds
  const double* a = nullptr;       // Adam elements of the exported block
  int32_t nbuf = 2;                // device buffers (= pinned staging buffers)
  double bw_h2d = 0, bw_d2h = 0;   // link bytes/s per direction
  double pack_rate = 0;            // bytes/s the worker pool packs (0: instant)
  double adam_rate = 0;            // Adam elements/s of the worker pool on an idle host (0: instant)
  double adam_bytes = 28;          // host memory bytes Adam moves per element
  double host_bw = 0;              // bytes/s host memory serves CPU and DMA together (0: unlimited)
  double chunk = 64.0 * (1 << 20); // bytes per packed chunk (its copy starts once it is packed)
};
struct SimOut {
  double period = 0;      // seconds between the starts of two steps' first computes
  double stall = 0;       // compute-stream idle seconds within that period
  double adam_busy = 0;   // seconds host Adam works within it
  double slab_wait = 0;   // seconds the driver waits for a free slab within it
  double pack = 0;        // seconds of packing on the driver's path within it
  double adam_rate = 0;   // Adam elements/s after the share DMA and packing take
};
// Simulates `steps` consecutive steps with K slabs and reports the last one;
// stall_v (n entries, may be null) receives the compute stream's wait before
// each visit of that step.  Adam's rate is the smaller of adam_rate and what
// host_bw leaves after the period's average DMA and pack traffic, found by
// fixed-point iteration over the period.
SimOut simulate(const SimIn& in, int32_t K, int32_t steps, double* stall_v);
// Chooses K in [k_min, k_max]: the shortest simulated period, then the
// fewest slabs within 0.5 % of it.
struct Plan {
  int32_t K = 1;
  SimOut out;
};
Plan plan(const SimIn& in, int32_t k_min, int32_t k_max);

}  // namespace mth
