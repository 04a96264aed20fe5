// fos_api.cu -- the C ABI of libfos_softmax.so (declared in include/fos_softmax.h).
//
// Host side only: argument validation, the choice of load path and launch geometry, the
// per-device set-up (SM count, shared-memory limit, kernel attributes, the address of the
// device error word) and the status strings.  None of these choices changes a result bit.
#include <cuda_occupancy.h>
#include <limits.h>
#include <stdint.h>

#include <cmath>
#include <map>
#include <mutex>
#include <tuple>

#include "fos_internal.h"

namespace fos {

// Device error word: a kernel whose bounded wait ran out stores kDevErrTimeout here.
__device__ unsigned g_device_error;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s
constexpr int kDefaultWarps = 8;

constexpr int kMaxStages = 16;
// The group forward: at most 15 groups per CTA (one named barrier each), 128 ring barriers in
// all, rings of at most 3 rows per group by default.
constexpr int kMaxGroups = 15;
constexpr int kGroupMaxBarriers = 128;
constexpr int kGroupDefaultMaxStages = 3;

struct DevInfo {
  bool ready = false;
  int index = 0;
  int sms = 0;
  int max_smem = 0;  // opt-in dynamic shared memory per block
  size_t smem_per_sm = 0;
  size_t reserved_smem = 0;  // shared memory the system keeps per block
  cudaOccDeviceProp occ;     // for residency counted on the host
  unsigned *err = nullptr;
};

DevInfo g_dev[kMaxDevices];
std::mutex g_mu;

fos_status device_info(DevInfo **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FOS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FOS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo &d = g_dev[dev];
  if (!d.ready) {
    d.index = dev;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return FOS_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FOS_ERR_CUDA;
    d.occ = cudaOccDeviceProp(prop);
    d.smem_per_sm = prop.sharedMemPerMultiprocessor;
    d.reserved_smem = prop.reservedSharedMemPerBlock;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return FOS_ERR_CUDA;
    d.err = static_cast<unsigned *>(p);
    const fos_dtype dts[3] = {FOS_F32, FOS_BF16, FOS_F16};
    for (fos_dtype dt : dts) {
      if (fwd_prepare(dt, d.max_smem) != cudaSuccess) return FOS_ERR_CUDA;
      if (bwd_prepare(dt, d.max_smem) != cudaSuccess) return FOS_ERR_CUDA;
    }
    d.ready = true;
  }
  *out = &d;
  return FOS_OK;
}

// The contractions encode TMA tensor maps (a driver call), which needs the device's context
// current in the calling thread.  A thread that has made no runtime call that binds it (the
// device index reads the same either way) can call in first: a PyTorch autograd worker thread,
// for one, whose first library call is a backward's QK contraction.  Setting the current device
// to itself binds its primary context; it changes nothing for a thread that already has it.
fos_status bind_context(const DevInfo &dev) {
  return cudaSetDevice(dev.index) == cudaSuccess ? FOS_OK : FOS_ERR_CUDA;
}

}  // namespace

int dtype_size(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return 4;
    case FOS_BF16: return 2;
    case FOS_F16: return 2;
  }
  return 0;
}

fos_status check_desc(const fos_desc *d) {
  if (d == nullptr) return FOS_ERR_INVALID;
  if (d->reserved != 0) return FOS_ERR_INVALID;
  if (d->rows < 0 || d->key_len < 1 || d->ld < d->key_len) return FOS_ERR_INVALID;
  if (d->causal != 0 && d->causal != 1) return FOS_ERR_INVALID;
  if (d->batch < 0 || d->heads < 0 || d->q_len < 0) return FOS_ERR_INVALID;
  const int64_t prod = (int64_t)d->batch * d->heads * d->q_len;
  if (prod != d->rows) return FOS_ERR_INVALID;
  if (d->causal && d->q_len > d->key_len) return FOS_ERR_INVALID;
  // rows * ld * 4 bytes must stay addressable
  if (d->rows > 0 && d->ld > (INT64_MAX / 8) / d->rows) return FOS_ERR_INVALID;
  return FOS_OK;
}

fos_status check_launch(const fos_launch *l) {
  if (l == nullptr) return FOS_OK;
  if (l->warps_per_cta < 0 || l->warps_per_cta > 16) return FOS_ERR_INVALID;
  if (l->ctas < 0) return FOS_ERR_INVALID;
  if (l->stages < 0 || l->stages > kMaxStages) return FOS_ERR_INVALID;
  if (l->load_path < 0 || l->load_path > 3) return FOS_ERR_INVALID;
  if (l->wait_timeout_ns < 0) return FOS_ERR_INVALID;
  if (l->test_stall != 0 && l->test_stall != 1) return FOS_ERR_INVALID;
  if (l->generic != 0 && l->generic != 1) return FOS_ERR_INVALID;
  if (l->groups_per_cta < 0 || l->groups_per_cta > 15) return FOS_ERR_INVALID;
  if (l->sink_fusion < 0 || l->sink_fusion > 2) return FOS_ERR_INVALID;
  return FOS_OK;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Resident CTAs per SM of a kernel instance at a block size and dynamic shared memory,
// memoised: a launch asks for up to eight ring depths and the answer never changes.
// `key` names the instance (kernel, dtype, tiles per warp, specialisation).
template <typename OccFn>
cudaError_t resident_ctas(int dev_index, uint32_t key, int threads, size_t smem, OccFn occ,
                          int *per_sm) {
  using Key = std::tuple<int, uint32_t, int, size_t>;
  static std::map<Key, int> memo;
  static std::mutex mu;
  const Key k{dev_index, key, threads, smem};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(k);
    if (it != memo.end()) {
      *per_sm = it->second;
      return cudaSuccess;
    }
  }
  cudaError_t e = occ(threads, smem, per_sm);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (memo.size() >= 4096) memo.clear();
  memo[k] = *per_sm;
  return cudaSuccess;
}

// CTAs per SM of a kernel whose code allocates tensor memory, `cols` columns per CTA (0: this
// launch allocates none), from its attributes, block size and dynamic shared memory.  The
// runtime's occupancy query counts such a kernel as filling its SM (the columns are allocated
// at run time), so the count comes from the occupancy calculator of cuda_occupancy.h at the
// full shared-memory carveout instead.  `fit` is that count; `per_sm` is it capped by the SM's
// 512 columns.
cudaError_t tmem_resident_ctas(const DevInfo &d, const cudaFuncAttributes &fa, int threads,
                               size_t smem, uint32_t cols, int *per_sm, int *fit = nullptr) {
  cudaOccFuncAttributes oa(fa);
  cudaOccDeviceState st;
  st.carveoutConfig = SHAREDMEM_CARVEOUT_MAX_SHARED;
  cudaOccResult r;
  if (cudaOccMaxActiveBlocksPerMultiprocessor(&r, &d.occ, &oa, &st, threads, smem) !=
      CUDA_OCC_SUCCESS)
    return cudaErrorInvalidValue;
  const int cap = cols ? (int)(kTmemColsPerSm / cols) : INT_MAX;
  if (fit) *fit = r.activeBlocksPerMultiprocessor;
  *per_sm = r.activeBlocksPerMultiprocessor < cap ? r.activeBlocksPerMultiprocessor : cap;
  return cudaSuccess;
}

// Dynamic shared memory for a tensor-memory launch: at least `smem`, and enough that no SM
// takes more CTAs than its columns serve (a CTA past that would wait in its allocation until
// another CTA of the launch exits).
cudaError_t tmem_pad_smem(const DevInfo &d, const cudaFuncAttributes &fa, int threads,
                          uint32_t cols, size_t *smem) {
  const int cap = (int)(kTmemColsPerSm / cols);
  for (int iter = 0; iter < 64; ++iter) {
    int per_sm = 0, fit = 0;
    cudaError_t e = tmem_resident_ctas(d, fa, threads, *smem, cols, &per_sm, &fit);
    if (e != cudaSuccess) return e;
    if (fit <= cap) return cudaSuccess;
    // the smallest footprint that leaves room for at most `cap` CTAs, then 128-byte steps
    const size_t want = d.smem_per_sm / (size_t)(cap + 1) + 1;
    const size_t used = d.reserved_smem + fa.sharedSizeBytes;
    size_t next = want > used ? want - used : 0;
    next = (next + 127) & ~(size_t)127;
    *smem = next > *smem ? next : *smem + 128;
    if (*smem > (size_t)d.max_smem) return cudaErrorInvalidValue;
  }
  return cudaErrorInvalidValue;
}

// Geometry of a row-kernel launch.
struct Plan {
  int threads = 0;
  int grid = 0;
  size_t smem = 0;
  int stages = 1;
  bool bulk = false;
};

// Fills the shared part of RowArgs and picks path, stages, CTAs.  `inputs` are the row
// arrays that are staged (scores, or P and dP); `copies` is how many of them a stage holds.
// seg_tiles > 0 plans a streaming kernel: stages hold segments of that many tiles (bulk
// copies only), the statistics arrays still cover the whole row.
template <typename OccFn>
fos_status plan_rows(const fos_desc *d, fos_dtype dt, int64_t row_base, int64_t nrows,
                     const void *const *inputs, int copies,
                     const void *output, const fos_launch *l, const DevInfo &dev,
                     size_t (*extra)(int, int), int default_warps, size_t stage_target,
                     uint32_t occ_key, OccFn occ, RowArgs *ra, Plan *pl, int seg_tiles = 0,
                     int extra_warps = 1) {
  const int esz = dtype_size(dt);
  const int T = (d->key_len + kTileK - 1) / kTileK;
  const int stage_tiles = (seg_tiles > 0 && seg_tiles < T) ? seg_tiles : T;
  const size_t stage_bytes = (size_t)stage_tiles * kTileK * esz;
  const bool stride16 = ((d->ld * esz) & 15) == 0;
  bool in_aligned = stride16;
  for (int i = 0; i < copies; ++i) in_aligned = in_aligned && aligned16(inputs[i]);
  const bool bulk_ok = in_aligned && (((int64_t)d->key_len * esz) & 15) == 0;
  const int path = l ? l->load_path : 0;
  const bool need_bulk = path == 1 || path == 3 || seg_tiles > 0;
  if (need_bulk && !bulk_ok) return FOS_ERR_UNSUPPORTED;
  if (seg_tiles > 0 && path == 2) return FOS_ERR_UNSUPPORTED;
  const bool bulk = need_bulk || (path == 0 && bulk_ok);

  const int warps = (l && l->warps_per_cta) ? l->warps_per_cta : default_warps;
  // the compute warps, one producer warp (and the streaming forward's merge warp)
  const int threads = (warps + extra_warps) * 32;
  const size_t slot = (size_t)copies * stage_bytes;
  const size_t fixed = extra(T, 0);
  if (fixed + slot > (size_t)dev.max_smem) return FOS_ERR_UNSUPPORTED;
  auto fits = [&](int n) { return fixed + (size_t)n * slot <= (size_t)dev.max_smem; };
  auto ctas_at = [&](int n, int *per_sm) {
    return resident_ctas(dev.index, occ_key, threads, fixed + (size_t)n * slot, occ, per_sm);
  };
  int stages = 1;
  if (bulk) {
    if (l && l->stages) {
      stages = l->stages;
      if (!fits(stages)) return FOS_ERR_UNSUPPORTED;
    } else if (fits(2)) {
      // The rows being computed, not the rows being copied, bound these kernels: take the
      // deepest ring (up to stage_target bytes, 8 rows) that keeps as many CTAs resident
      // per SM as a two-row ring does.
      int cap = (int)(stage_target / slot);
      cap = cap < 2 ? 2 : (cap > 8 ? 8 : cap);
      while (cap > 2 && !fits(cap)) --cap;
      int base = 0;
      if (ctas_at(2, &base) != cudaSuccess) return FOS_ERR_CUDA;
      stages = 2;
      for (int n = cap; n > 2; --n) {
        int c = 0;
        if (ctas_at(n, &c) != cudaSuccess) return FOS_ERR_CUDA;
        if (c >= base) {
          stages = n;
          break;
        }
      }
    }
  }
  const size_t smem = fixed + stages * slot;

  int grid = 0;
  if (l && l->ctas) {
    grid = l->ctas;
  } else {
    int per_sm = 0;
    if (ctas_at(stages, &per_sm) != cudaSuccess) return FOS_ERR_CUDA;
    if (per_sm < 1) return FOS_ERR_UNSUPPORTED;
    grid = per_sm * dev.sms;
  }
  if ((int64_t)grid > nrows) grid = (int)nrows;

  ra->rows = nrows;
  ra->row_base = row_base;
  ra->ld = d->ld;
  ra->L = d->key_len;
  ra->heads = d->heads;
  ra->q_len = d->q_len;
  ra->causal = d->causal;
  ra->kv_valid_len = d->kv_valid_len;
  ra->key_mask = d->key_mask;
  ra->T = T;
  ra->stages = stages;
  ra->stage_bytes = (uint32_t)stage_bytes;
  ra->seg_tiles = seg_tiles > 0 ? stage_tiles : 0;
  ra->use_bulk = bulk ? 1 : 0;
  ra->in_vec = in_aligned ? 1 : 0;
  ra->out_vec = (stride16 && aligned16(output)) ? 1 : 0;
  ra->timeout_ns = (l && l->wait_timeout_ns) ? (uint64_t)l->wait_timeout_ns : kDefaultTimeoutNs;
  ra->test_stall = l ? l->test_stall : 0;
  ra->need_geo = (d->causal || d->kv_valid_len || d->key_mask) ? 1 : 0;
  ra->geo32 = (row_base + nrows <= (int64_t)INT32_MAX) ? 1 : 0;
  ra->qdiv = make_fastdiv((uint32_t)d->q_len);
  ra->hdiv = make_fastdiv((uint32_t)d->heads);
  ra->err = dev.err;

  pl->threads = threads;
  pl->grid = grid;
  pl->smem = smem;
  pl->stages = stages;
  pl->bulk = bulk;
  return FOS_OK;
}

}  // namespace
}  // namespace fos

using namespace fos;

namespace fos {

// Rows longer than a shared-memory stage (or load_path 3) are read twice in segments of
// max(16, 2 x warps) tiles, so that every warp takes two tiles of a full segment.  Default
// launches, measured on GB300 (1,024 rows of 262,144 bf16 keys; 8 / 12 / 16 / 24 / 31 compute
// warps, 152 / 304 / 456 CTAs, rings of 2..6 segments; same bits throughout): the forward
// recomputes its exponentials and is issue-bound, best with 12 warps, two CTAs per SM and six
// segments in flight (328 us; 340 with 8 warps and three); the backward is bound by DRAM and
// runs fastest with 16 warps, one CTA per SM and four segments (377 us; 400 with 8 warps):
// fewer rows in flight leave more of each row in L2 for its second read.  Rows whose tile
// statistics leave no room for that ring fall back to 8 warps and 16-tile segments.
constexpr int kStreamSegTiles = 16;
constexpr int kStreamWarpsFwd = 12;
constexpr int kStreamStagesFwd = 6;
constexpr int kStreamWarpsBwd = 16;
constexpr int kStreamStagesBwd = 4;
constexpr int kStreamWarpsNarrow = 8;

int stream_seg_tiles(int warps) {
  return 2 * warps > kStreamSegTiles ? 2 * warps : kStreamSegTiles;
}

// The ring bytes plan_rows may fill for a streaming launch: `stages` segments.
size_t stream_ring_target(int seg_tiles, fos_dtype dt, int copies, int stages) {
  return (size_t)stages * copies * seg_tiles * kTileK * dtype_size(dt);
}

bool stream_rows(const fos_desc *desc, fos_dtype dtype, int copies, size_t (*extra)(int, int),
                 const fos_launch *launch, const DevInfo &dev) {
  if (launch && launch->load_path == 3) return true;
  const int T = (desc->key_len + kTileK - 1) / kTileK;
  const size_t whole = extra(T, 0) + (size_t)copies * T * kTileK * dtype_size(dtype);
  return whole > (size_t)dev.max_smem;
}

// Rows of at most this many tiles go to the one-warp-per-row forward kernel by default: eight
// warps per CTA with one row buffer each (measured on GB300 against 2 / 4 warps and 1..3
// buffers: 3-7 % faster over 256..2048 keys).
constexpr int kRowWarpMaxTiles = 8;
constexpr int kRowWarpWarps = 8;
constexpr int kRowWarpStages = 1;
// The backward holds a buffer until dScores are written: one buffer per warp lets twice the warps
// reside, which hides each warp's copy better than a second buffer (measured: 336 vs 398 us on
// the causal sink workload).
constexpr int kRowWarpStagesBwd = 1;
constexpr int kRowWarpWarpsBwd = 4;

// Row arguments of a one-warp-per-row launch (bulk copies, whole rows per buffer).
void fill_rowwarp_args(const fos_desc *desc, int esz, int64_t row_base, int64_t nrows, int T,
                       int stages, size_t stage_bytes, const void *output,
                       const fos_launch *launch, const DevInfo &dev, RowArgs *a) {
  a->rows = nrows;
  a->row_base = row_base;
  a->ld = desc->ld;
  a->L = desc->key_len;
  a->heads = desc->heads;
  a->q_len = desc->q_len;
  a->causal = desc->causal;
  a->kv_valid_len = desc->kv_valid_len;
  a->key_mask = desc->key_mask;
  a->T = T;
  a->stages = stages;
  a->stage_bytes = (uint32_t)stage_bytes;
  a->seg_tiles = 0;
  a->use_bulk = 1;
  a->in_vec = 1;
  a->out_vec = (((desc->ld * esz) & 15) == 0 && aligned16(output)) ? 1 : 0;
  a->timeout_ns = (launch && launch->wait_timeout_ns) ? (uint64_t)launch->wait_timeout_ns
                                                      : kDefaultTimeoutNs;
  a->test_stall = launch ? launch->test_stall : 0;
  a->need_geo = (desc->causal || desc->kv_valid_len || desc->key_mask) ? 1 : 0;
  a->geo32 = (row_base + nrows <= (int64_t)INT32_MAX) ? 1 : 0;
  a->qdiv = make_fastdiv((uint32_t)desc->q_len);
  a->hdiv = make_fastdiv((uint32_t)desc->heads);
  a->err = dev.err;
}

// The one-warp-per-row forward: needs bulk copies (FOS_ERR_UNSUPPORTED otherwise, so the
// caller can fall back to the CTA kernel with plain loads).
fos_status run_fwd_rowwarp(const fos_desc *desc, fos_dtype dtype, int64_t row_base, int64_t nrows,
                           const void *scores, void *probs, float *lse, cudaStream_t stream,
                           const fos_launch *launch, const DevInfo &dev) {
  const int esz = dtype_size(dtype);
  const int T = (desc->key_len + kTileK - 1) / kTileK;
  const bool bulk_ok = aligned16(scores) && ((desc->ld * esz) & 15) == 0 &&
                       (((int64_t)desc->key_len * esz) & 15) == 0;
  if (!bulk_ok) return FOS_ERR_UNSUPPORTED;
  const int kt = T <= 2 ? 2 : (T <= 4 ? 4 : 8);
  const int warps = (launch && launch->warps_per_cta) ? launch->warps_per_cta : kRowWarpWarps;
  int stages = (launch && launch->stages) ? launch->stages : kRowWarpStages;
  if (warps * stages > 16) stages = 16 / warps > 0 ? 16 / warps : 1;  // 16 barrier slots
  if (warps * stages > 16) return FOS_ERR_UNSUPPORTED;
  const size_t stage_bytes = (size_t)T * kTileK * esz;
  size_t smem = fwd_rowwarp_smem(warps, stages, stage_bytes);
  if (smem > (size_t)dev.max_smem) return FOS_ERR_UNSUPPORTED;
  const int threads = warps * 32;
  // e_j are parked in tensor memory: residency counted here, shared memory padded so that no
  // SM takes more CTAs than it has columns for (see tmem_resident_ctas)
  const uint32_t cols = kt > 2 ? fwd_tmem_cols(warps, kt) : 0u;  // kt 2: registers
  cudaFuncAttributes fa;
  if (fwd_rowwarp_attributes(dtype, kt, &fa) != cudaSuccess) return FOS_ERR_CUDA;
  if (cols && tmem_pad_smem(dev, fa, threads, cols, &smem) != cudaSuccess)
    return FOS_ERR_UNSUPPORTED;
  int grid = 0;
  if (launch && launch->ctas) {
    grid = launch->ctas;
  } else {
    int per_sm = 0;
    if (resident_ctas(dev.index, 0x500u | ((uint32_t)dtype << 4) | (uint32_t)kt | (cols << 8),
                      threads, smem,
                      [&dev, &fa, cols](int th, size_t sm, int *n) {
                        return tmem_resident_ctas(dev, fa, th, sm, cols, n);
                      },
                      &per_sm) != cudaSuccess)
      return FOS_ERR_CUDA;
    if (per_sm < 1) return FOS_ERR_UNSUPPORTED;
    grid = per_sm * dev.sms;
  }
  const int64_t need = (nrows + warps - 1) / warps;  // CTAs with at least one row
  if ((int64_t)grid > need) grid = (int)need;

  FwdArgs a{};
  fill_rowwarp_args(desc, esz, row_base, nrows, T, stages, stage_bytes, probs, launch, dev, &a);
  if (desc->sink) a.need_geo = 1;  // the merge needs the row's head
  a.scores = scores;
  a.probs = probs;
  a.lse = lse;
  a.sink = desc->sink;
  a.keep_e = 1;
  a.tmem_cols = cols;
  if (fwd_rowwarp_launch(dtype, kt, a, grid, threads, smem, stream) != cudaSuccess)
    return FOS_ERR_CUDA;
  return FOS_OK;
}

// The group forward (several row groups of `nw` warps per CTA, kt tiles parked per warp, no
// producer warp): needs bulk copies (FOS_ERR_UNSUPPORTED otherwise, so the caller can fall back
// to the CTA kernel with plain loads).  Groups per CTA and ring depth are chosen for the most
// rows in flight per SM (registers, tensor-memory columns and shared memory all bound it), then
// the deeper ring, then the smaller CTA.
fos_status run_fwd_group(const fos_desc *desc, fos_dtype dtype, int64_t row_base, int64_t nrows,
                         const void *scores, void *probs, float *lse, cudaStream_t stream,
                         const fos_launch *launch, const DevInfo &dev, int nw, int kt,
                         bool fast) {
  const int esz = dtype_size(dtype);
  const int T = (desc->key_len + kTileK - 1) / kTileK;
  const bool bulk_ok = aligned16(scores) && ((desc->ld * esz) & 15) == 0 &&
                       (((int64_t)desc->key_len * esz) & 15) == 0;
  if (!bulk_ok) return FOS_ERR_UNSUPPORTED;
  fast = fast && ((desc->ld * esz) & 15) == 0 && aligned16(probs);
  const size_t stage_bytes = (size_t)T * kTileK * esz;
  cudaFuncAttributes fa;
  if (fwd_group_attributes(dtype, kt, fast, &fa) != cudaSuccess) return FOS_ERR_CUDA;
  const int max_g = 32 / nw < kMaxGroups ? 32 / nw : kMaxGroups;  // 1024 threads, 15 barriers
  const int g_lo = (launch && launch->groups_per_cta) ? launch->groups_per_cta : 1;
  const int g_hi = (launch && launch->groups_per_cta) ? launch->groups_per_cta : max_g;
  const int s_lo = (launch && launch->stages) ? launch->stages : 1;
  const int s_hi = (launch && launch->stages) ? launch->stages : kGroupDefaultMaxStages;
  if (g_hi * nw > 32 || g_hi > kMaxGroups || g_lo * s_lo > kGroupMaxBarriers)
    return FOS_ERR_UNSUPPORTED;
  int best_g = 0, best_ns = 0, best_rows = 0, best_per = 0;
  uint32_t best_cols = 0;
  size_t best_smem = 0;
  for (int ng = g_lo; ng <= g_hi; ++ng) {
    const uint32_t cols = fwd_tmem_cols(ng * nw, kt);
    if (cols > kTmemColsPerSm) continue;
    for (int ns = s_lo; ns <= s_hi; ++ns) {
      if (ng * ns > kGroupMaxBarriers) continue;
      const size_t smem = fwd_group_smem(ng, ns, stage_bytes, T);
      if (smem > (size_t)dev.max_smem) continue;
      int per_sm = 0;
      if (tmem_resident_ctas(dev, fa, ng * nw * 32, smem, cols, &per_sm) != cudaSuccess)
        return FOS_ERR_CUDA;
      const int rows = ng * per_sm;
      // the most rows in flight; then the fewest CTAs per SM (more groups per CTA: measured
      // 2-10 % faster at equal rows in flight on 17- to 32-tile rows); then the deeper ring
      if (rows > best_rows || (rows == best_rows && per_sm < best_per) ||
          (rows == best_rows && per_sm == best_per && ns > best_ns)) {
        best_rows = rows;
        best_g = ng;
        best_ns = ns;
        best_per = per_sm;
        best_cols = cols;
        best_smem = smem;
      }
    }
  }
  if (best_rows < 1) return FOS_ERR_UNSUPPORTED;
  const int threads = best_g * nw * 32;
  size_t smem = best_smem;
  if (tmem_pad_smem(dev, fa, threads, best_cols, &smem) != cudaSuccess) return FOS_ERR_UNSUPPORTED;
  int grid = (launch && launch->ctas) ? launch->ctas : best_per * dev.sms;
  const int64_t need = (nrows + best_g - 1) / best_g;  // CTAs with at least one row
  if ((int64_t)grid > need) grid = (int)need;

  FwdArgs a{};
  fill_rowwarp_args(desc, esz, row_base, nrows, T, best_ns, stage_bytes, probs, launch, dev, &a);
  if (desc->sink) a.need_geo = 1;  // the merge needs the row's head
  a.scores = scores;
  a.probs = probs;
  a.lse = lse;
  a.sink = desc->sink;
  a.keep_e = 1;
  a.tmem_cols = best_cols;
  a.group_warps = nw;
  if (fwd_group_launch(dtype, kt, fast, a, grid, threads, smem, stream) != cudaSuccess)
    return FOS_ERR_CUDA;
  return FOS_OK;
}

fos_status run_fwd(const fos_desc *desc, fos_dtype dtype, int64_t row_base, int64_t nrows,
                   const void *scores, void *probs, float *lse, cudaStream_t stream,
                   const fos_launch *launch) {
  DevInfo *dev = nullptr;
  fos_status st = device_info(&dev);
  if (st != FOS_OK) return st;

  FwdArgs a{};
  Plan pl;
  const void *inputs[1] = {scores};
  if (stream_rows(desc, dtype, 1, fwd_extra_smem, launch, *dev)) {
    const bool given = launch && launch->warps_per_cta;
    auto plan = [&](int warps) {
      const int seg = stream_seg_tiles(warps);
      return plan_rows(desc, dtype, row_base, nrows, inputs, 1, probs, launch, *dev,
                       fwd_stream_extra_smem, warps,
                       stream_ring_target(seg, dtype, 1, kStreamStagesFwd),
                       0x300u | ((uint32_t)dtype << 4),
                       [dtype](int th, size_t sm, int *n) {
                         return fwd_stream_occupancy(dtype, th, sm, n);
                       },
                       &a, &pl, seg, 2);
    };
    st = plan(given ? launch->warps_per_cta : kStreamWarpsFwd);
    if (st == FOS_ERR_UNSUPPORTED && !given) st = plan(kStreamWarpsNarrow);
    if (st != FOS_OK) return st;
    a.scores = scores;
    a.probs = probs;
    a.lse = lse;
    a.sink = desc->sink;
    if (desc->sink) a.need_geo = 1;
    if (fwd_stream_launch(dtype, a, pl.grid, pl.threads, pl.smem, stream) != cudaSuccess)
      return FOS_ERR_CUDA;
    return FOS_OK;
  }
  const int T = (desc->key_len + kTileK - 1) / kTileK;
  if (T <= kRowWarpMaxTiles && !(launch && (launch->generic || launch->load_path == 2))) {
    st = run_fwd_rowwarp(desc, dtype, row_base, nrows, scores, probs, lse, stream, launch, *dev);
    if (st != FOS_ERR_UNSUPPORTED || (launch && launch->load_path == 1)) return st;
    // unaligned rows: the CTA kernel with plain loads
  }
  // fp32 rows of 25..32 tiles: four tiles per warp and one row buffer per CTA measured 5 %
  // faster than the bf16-fitted default (8192 keys on GB300)
  const bool f32_mid = dtype == FOS_F32 && T > 24 && T <= 32;
  const int warps = (launch && launch->warps_per_cta) ? launch->warps_per_cta
                                                      : (f32_mid ? (T + 3) / 4 : fwd_default_warps(T));
  fos_launch tuned{};
  const fos_launch *lp = launch;
  if (f32_mid && !(launch && (launch->warps_per_cta || launch->stages))) {
    if (launch) tuned = *launch;
    tuned.stages = 1;
    lp = &tuned;
  }
  int kt = fwd_tiles_per_warp(T, warps);
  const bool in_regs = T <= warps * kt;
  if (!in_regs) kt = 2;  // e_j are recomputed: keep the register footprint small
  // The specialised instance covers the common case; the generic one covers the rest.
  const int esz = dtype_size(dtype);
  const bool fast = in_regs && !(launch && launch->generic) && !(launch && launch->load_path == 2) &&
                    !desc->causal && !desc->kv_valid_len && !desc->key_mask && !desc->sink &&
                    aligned16(scores) && aligned16(probs) && ((desc->ld * esz) & 15) == 0 &&
                    (((int64_t)desc->key_len * esz) & 15) == 0;
  // Every warp parks its tiles in tensor memory: the group kernel, unless the general CTA
  // kernel or plain loads are asked for (or the rows do not allow bulk copies).  fp32 rows of
  // 25..32 tiles keep their tuned CTA launch (measured faster there) unless groups are asked
  // for.
  const bool groups_asked = launch && launch->groups_per_cta;
  if (in_regs && kt >= 4 && !(launch && (launch->generic || launch->load_path == 2)) &&
      (!f32_mid || groups_asked)) {
    st = run_fwd_group(desc, dtype, row_base, nrows, scores, probs, lse, stream, launch, *dev,
                       warps, kt, fast);
    if (st != FOS_ERR_UNSUPPORTED || (launch && launch->load_path == 1)) return st;
  }
  if (launch && launch->groups_per_cta) return FOS_ERR_UNSUPPORTED;  // only the group kernel
  // Parked e_j take tensor-memory columns; residency is then counted here (see
  // tmem_resident_ctas) and shared memory padded so that no SM takes more CTAs than it has
  // columns for.
  const uint32_t cols = (in_regs && kt > 2) ? fwd_tmem_cols(warps, kt) : 0u;
  cudaFuncAttributes fa;
  if (fwd_attributes(dtype, kt, fast, &fa) != cudaSuccess) return FOS_ERR_CUDA;
  // ring of up to 24 KB per CTA: rows are consumed right after their tile pass
  const uint32_t key = 0x100u | ((uint32_t)dtype << 4) | ((uint32_t)kt << 1) | (fast ? 1u : 0u);
  const DevInfo &dv = *dev;
  st = plan_rows(desc, dtype, row_base, nrows, inputs, 1, probs, lp, *dev, fwd_extra_smem,
                 warps, 24 * 1024, key | (cols << 8),
                 [cols, &fa, &dv](int th, size_t sm, int *n) {
                   return tmem_resident_ctas(dv, fa, th, sm, cols, n);
                 },
                 &a, &pl);
  if (st != FOS_OK) return st;
  if (cols && tmem_pad_smem(*dev, fa, pl.threads, cols, &pl.smem) != cudaSuccess)
    return FOS_ERR_UNSUPPORTED;
  a.keep_e = in_regs ? 1 : 0;
  a.scores = scores;
  a.probs = probs;
  a.lse = lse;
  a.sink = desc->sink;
  a.tmem_cols = cols;
  if (desc->sink) a.need_geo = 1;  // the merge needs the row's head
  if (fwd_launch(dtype, kt, fast && a.use_bulk && a.out_vec, a, pl.grid, pl.threads, pl.smem,
                 stream) != cudaSuccess)
    return FOS_ERR_CUDA;
  return FOS_OK;
}

// The sink gradient fused into the backward: octet layout of the problem's positions and the
// arrays the kernels read (lse) and write (the octet sums).
void fill_octets(const fos_desc *d, const float *lse, float *oct_sums, BwdArgs *a) {
  a->lse = lse;
  a->sink = d->sink;
  a->oct_sums = oct_sums;
  a->pos_end = (int64_t)d->batch * d->q_len;
  a->oct_per_head = (a->pos_end + 7) / 8;
  a->octdiv = make_fastdiv((uint32_t)(a->oct_per_head > 0 && a->oct_per_head < ((int64_t)1 << 32)
                                          ? a->oct_per_head
                                          : 1));
  a->oct32 = ((int64_t)d->heads * a->oct_per_head < ((int64_t)1 << 32) &&
              a->pos_end < ((int64_t)1 << 32))
                 ? 1
                 : 0;
}

// The one-warp-per-row backward for rows of at most kRowWarpMaxTiles tiles: needs bulk copies
// of P and dP (FOS_ERR_UNSUPPORTED otherwise, so the caller can fall back to the CTA kernel).
fos_status run_bwd_rowwarp(const fos_desc *desc, fos_dtype dtype, int64_t row_base, int64_t nrows,
                           const void *probs, const void *dprobs, void *dscores, float *delta,
                           cudaStream_t stream, const fos_launch *launch, const DevInfo &dev,
                           const float *lse = nullptr, float *oct_sums = nullptr) {
  const int esz = dtype_size(dtype);
  const int T = (desc->key_len + kTileK - 1) / kTileK;
  const bool bulk_ok = aligned16(probs) && aligned16(dprobs) && ((desc->ld * esz) & 15) == 0 &&
                       (((int64_t)desc->key_len * esz) & 15) == 0;
  if (!bulk_ok) return FOS_ERR_UNSUPPORTED;
  const int warps = (launch && launch->warps_per_cta) ? launch->warps_per_cta : kRowWarpWarpsBwd;
  int stages = (launch && launch->stages) ? launch->stages : kRowWarpStagesBwd;
  if (warps * stages > 16) stages = 16 / warps > 0 ? 16 / warps : 1;  // 16 barrier slots
  if (warps * stages > 16) return FOS_ERR_UNSUPPORTED;
  const size_t stage_bytes = (size_t)T * kTileK * esz;
  const size_t smem = bwd_rowwarp_smem(warps, stages, stage_bytes, T);
  if (smem > (size_t)dev.max_smem) return FOS_ERR_UNSUPPORTED;
  const int threads = warps * 32;
  int grid = 0;
  if (launch && launch->ctas) {
    grid = launch->ctas;
  } else {
    int per_sm = 0;
    if (resident_ctas(dev.index, 0x600u | ((uint32_t)dtype << 4), threads, smem,
                      [dtype](int th, size_t sm, int *n) {
                        return bwd_rowwarp_occupancy(dtype, th, sm, n);
                      },
                      &per_sm) != cudaSuccess)
      return FOS_ERR_CUDA;
    if (per_sm < 1) return FOS_ERR_UNSUPPORTED;
    grid = per_sm * dev.sms;
  }
  const int64_t need = (nrows + warps - 1) / warps;  // CTAs with at least one row
  if ((int64_t)grid > need) grid = (int)need;

  BwdArgs a{};
  fill_rowwarp_args(desc, esz, row_base, nrows, T, stages, stage_bytes, dscores, launch, dev, &a);
  a.probs = probs;
  a.dprobs = dprobs;
  a.dscores = dscores;
  a.delta = delta;
  if (oct_sums) fill_octets(desc, lse, oct_sums, &a);
  if (bwd_rowwarp_launch(dtype, a, grid, threads, smem, stream, oct_sums != nullptr) !=
      cudaSuccess)
    return FOS_ERR_CUDA;
  return FOS_OK;
}

fos_status run_bwd(const fos_desc *desc, fos_dtype dtype, int64_t row_base, int64_t nrows,
                   const void *probs, const void *dprobs, void *dscores, float *delta,
                   cudaStream_t stream, const fos_launch *launch, const float *lse,
                   float *oct_sums, bool *fused) {
  DevInfo *dev = nullptr;
  fos_status st = device_info(&dev);
  if (st != FOS_OK) return st;
  if (fused) *fused = false;

  BwdArgs a{};
  Plan pl;
  const void *inputs[2] = {probs, dprobs};
  if (stream_rows(desc, dtype, 2, bwd_extra_smem, launch, *dev)) {
    const bool given = launch && launch->warps_per_cta;
    auto plan = [&](int warps) {
      const int seg = stream_seg_tiles(warps);
      return plan_rows(desc, dtype, row_base, nrows, inputs, 2, dscores, launch, *dev,
                       bwd_extra_smem, warps,
                       stream_ring_target(seg, dtype, 2, kStreamStagesBwd),
                       0x400u | ((uint32_t)dtype << 4),
                       [dtype](int th, size_t sm, int *n) {
                         return bwd_stream_occupancy(dtype, th, sm, n);
                       },
                       &a, &pl, seg);
    };
    st = plan(given ? launch->warps_per_cta : kStreamWarpsBwd);
    if (st == FOS_ERR_UNSUPPORTED && !given) st = plan(kStreamWarpsNarrow);
    if (st != FOS_OK) return st;
    a.probs = probs;
    a.dprobs = dprobs;
    a.dscores = dscores;
    // no octets on this path: with a sink gradient to come, delta goes to the workspace
    a.delta = (delta == nullptr && oct_sums) ? oct_sums : delta;
    if (bwd_stream_launch(dtype, a, pl.grid, pl.threads, pl.smem, stream) != cudaSuccess)
      return FOS_ERR_CUDA;
    return FOS_OK;
  }
  if ((desc->key_len + kTileK - 1) / kTileK <= kRowWarpMaxTiles &&
      !(launch && (launch->generic || launch->load_path == 2))) {
    // With a sink gradient to come, the one-warp kernel takes octets only when asked: the two
    // launches (delta to the workspace, then the sink-gradient kernel) measured 10 % faster on
    // short causal rows (343 against 381 us on 2 x 64 heads x 2,048 queries), with the same bits.
    const bool fuse_rw = oct_sums != nullptr && launch && launch->sink_fusion == 1;
    float *rw_delta = (oct_sums != nullptr && !fuse_rw && delta == nullptr) ? oct_sums : delta;
    st = run_bwd_rowwarp(desc, dtype, row_base, nrows, probs, dprobs, dscores, rw_delta, stream,
                         launch, *dev, lse, fuse_rw ? oct_sums : nullptr);
    if (st == FOS_OK && fused) *fused = fuse_rw;
    if (st != FOS_ERR_UNSUPPORTED || (launch && launch->load_path == 1)) return st;
    // unaligned rows: the CTA kernel with plain loads
  }
  const int esz = dtype_size(dtype);
  const bool fast = !(launch && launch->generic) && !(launch && launch->load_path == 2) &&
                    !desc->causal && !desc->kv_valid_len && !desc->key_mask &&
                    aligned16(probs) && aligned16(dprobs) && aligned16(dscores) &&
                    ((desc->ld * esz) & 15) == 0 && (((int64_t)desc->key_len * esz) & 15) == 0;
  st = plan_rows(desc, dtype, row_base, nrows, inputs, 2, dscores, launch, *dev, bwd_extra_smem,
                 bwd_default_warps((desc->key_len + kTileK - 1) / kTileK), 48 * 1024,
                 0x200u | ((uint32_t)dtype << 4) | (fast ? 1u : 0u),
                 [dtype, fast](int th, size_t sm, int *n) {
                   return bwd_occupancy(dtype, fast, th, sm, n);
                 },
                 &a, &pl);
  if (st != FOS_OK) return st;
  a.probs = probs;
  a.dprobs = dprobs;
  a.dscores = dscores;
  a.delta = delta;
  // The sink gradient rides along when there are enough octets to keep every CTA busy (each
  // CTA then takes whole octets; with few of them the grid would idle).  Measured against the
  // two launches on rows of 4,352 and 4,608 keys: within 1.3 % either way, the same bits.
  bool fuse = false;
  if (oct_sums) {
    fill_octets(desc, lse, oct_sums, &a);
    fuse = (int64_t)desc->heads * a.oct_per_head >= 4 * (int64_t)pl.grid &&
           !(launch && launch->sink_fusion == 2);
    if (!fuse) {  // delta then goes to the workspace for the sink-gradient kernel
      a.oct_sums = nullptr;
      if (delta == nullptr) a.delta = oct_sums;
    }
  }
  if (bwd_launch(dtype, fast && a.use_bulk && a.out_vec, a, pl.grid, pl.threads, pl.smem, stream,
                 fuse) != cudaSuccess)
    return FOS_ERR_CUDA;
  if (fused) *fused = fuse;
  return FOS_OK;
}

fos_status run_sink(const fos_desc *desc, const float *lse, const float *delta, float *d_sink,
                    cudaStream_t stream, const fos_launch *launch) {
  DevInfo *dev = nullptr;
  fos_status st = device_info(&dev);
  if (st != FOS_OK) return st;
  SinkArgs a{};
  fill_sink_args(desc, &a);
  a.lse = lse;
  a.delta = delta;
  a.d_sink = d_sink;
  const int warps = (launch && launch->warps_per_cta) ? launch->warps_per_cta : kDefaultWarps;
  if (sink_launch(a, warps * 32, stream) != cudaSuccess) return FOS_ERR_CUDA;
  return FOS_OK;
}

}  // namespace fos

extern "C" fos_status fos_softmax_fwd(const fos_desc *desc, fos_dtype dtype, const void *scores,
                                      void *probs, float *lse, cudaStream_t stream,
                                      const fos_launch *launch) {
  fos_status st = check_desc(desc);
  if (st != FOS_OK) return st;
  if ((st = check_launch(launch)) != FOS_OK) return st;
  if (dtype_size(dtype) == 0) return FOS_ERR_INVALID;
  if (desc->rows == 0) return FOS_OK;  // nothing to do; empty buffers may be null
  if (scores == nullptr || probs == nullptr || lse == nullptr) return FOS_ERR_INVALID;
  return run_fwd(desc, dtype, 0, desc->rows, scores, probs, lse, stream, launch);
}

extern "C" fos_status fos_softmax_bwd(const fos_desc *desc, fos_dtype dtype, const void *probs,
                                      const void *dprobs, void *dscores, float *delta,
                                      cudaStream_t stream, const fos_launch *launch) {
  fos_status st = check_desc(desc);
  if (st != FOS_OK) return st;
  if ((st = check_launch(launch)) != FOS_OK) return st;
  if (dtype_size(dtype) == 0) return FOS_ERR_INVALID;
  if (desc->rows == 0) return FOS_OK;  // nothing to do; empty buffers may be null
  if (probs == nullptr || dprobs == nullptr || dscores == nullptr) return FOS_ERR_INVALID;
  return run_bwd(desc, dtype, 0, desc->rows, probs, dprobs, dscores, delta, stream, launch);
}

extern "C" size_t fos_bwd_sink_workspace_bytes(const fos_desc *desc) {
  if (check_desc(desc) != FOS_OK) return 0;
  const int64_t octets = (int64_t)desc->heads * (((int64_t)desc->batch * desc->q_len + 7) / 8);
  const int64_t n = desc->rows > octets ? desc->rows : octets;
  return ((size_t)n * sizeof(float) + 255) & ~(size_t)255;
}

extern "C" fos_status fos_softmax_bwd_sink(const fos_desc *desc, fos_dtype dtype,
                                           const void *probs, const void *dprobs, void *dscores,
                                           float *delta, const float *lse, float *d_sink,
                                           void *workspace, size_t workspace_bytes,
                                           cudaStream_t stream, const fos_launch *launch) {
  fos_status st = check_desc(desc);
  if (st != FOS_OK) return st;
  if ((st = check_launch(launch)) != FOS_OK) return st;
  if (dtype_size(dtype) == 0) return FOS_ERR_INVALID;
  if (desc->sink == nullptr || d_sink == nullptr) return FOS_ERR_INVALID;
  if (desc->heads == 0) return FOS_OK;
  const size_t need = fos_bwd_sink_workspace_bytes(desc);
  if (desc->rows > 0 && (probs == nullptr || dprobs == nullptr || dscores == nullptr ||
                         lse == nullptr || workspace == nullptr || workspace_bytes < need ||
                         !aligned16(workspace)))
    return FOS_ERR_INVALID;
  float *ws = static_cast<float *>(workspace);
  bool fused = false;
  if (desc->rows > 0) {
    // the workspace takes the octet sums, or delta (when none was given) if the rows go to a
    // kernel that takes no octets; the sink-gradient kernel then follows (same bits)
    st = run_bwd(desc, dtype, 0, desc->rows, probs, dprobs, dscores, delta, stream, launch, lse,
                 ws, &fused);
    if (st != FOS_OK) return st;
  }
  if (fused) {
    DevInfo *dev = nullptr;
    if ((st = device_info(&dev)) != FOS_OK) return st;
    SinkArgs a{};
    fill_sink_args(desc, &a);
    a.d_sink = d_sink;
    const int warps = (launch && launch->warps_per_cta) ? launch->warps_per_cta : kDefaultWarps;
    if (sink_merge_launch(a, ws, ((int64_t)desc->batch * desc->q_len + 7) / 8, warps * 32,
                          stream) != cudaSuccess)
      return FOS_ERR_CUDA;
    return FOS_OK;
  }
  return run_sink(desc, lse, delta ? delta : ws, d_sink, stream, launch);
}

extern "C" fos_status fos_qk_scores(const fos_qk_desc *desc, fos_dtype in_dtype,
                                     fos_dtype out_dtype, const void *q, const void *k,
                                     void *scores, cudaStream_t stream) {
  if (desc == nullptr) return FOS_ERR_INVALID;
  if (desc->tile_n != 0 && desc->tile_n != 128 && desc->tile_n != 256) return FOS_ERR_INVALID;
  const fos_qk_desc &d = *desc;
  if (d.batch < 0 || d.q_heads < 0 || d.kv_heads < 1 || d.q_len < 0 || d.kv_len < 0 ||
      d.head_dim < 1 || d.ld_scores < d.kv_len || d.q_heads % d.kv_heads != 0)
    return FOS_ERR_INVALID;
  if (in_dtype != FOS_BF16 && in_dtype != FOS_F16) return FOS_ERR_INVALID;
  if (out_dtype != FOS_F32 && out_dtype != FOS_BF16 && out_dtype != FOS_F16) return FOS_ERR_INVALID;
  if ((int64_t)d.batch * d.q_heads * d.q_len * d.kv_len == 0) return FOS_OK;
  if (q == nullptr || k == nullptr || scores == nullptr) return FOS_ERR_INVALID;
  if (d.head_dim != 64 && d.head_dim != 128) return FOS_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(scores) ||
      ((d.ld_scores * dtype_size(out_dtype)) & 15) != 0)
    return FOS_ERR_UNSUPPORTED;
  if ((int64_t)d.batch * d.q_heads > 65535 || (d.q_len + 127) / 128 > 65535)
    return FOS_ERR_UNSUPPORTED;
  DevInfo *dev = nullptr;
  fos_status st = device_info(&dev);
  if (st != FOS_OK) return st;
  if ((st = bind_context(*dev)) != FOS_OK) return st;
  return run_qk(desc, in_dtype, out_dtype, q, k, scores, stream, dev->err, dev->max_smem,
                dev->sms);
}

extern "C" fos_status fos_pv_out(const fos_pv_desc *desc, fos_dtype in_dtype,
                                  fos_dtype out_dtype, const void *probs, const void *v,
                                  void *out, cudaStream_t stream) {
  if (desc == nullptr) return FOS_ERR_INVALID;
  const fos_pv_desc &d = *desc;
  if (d.batch < 0 || d.q_heads < 0 || d.kv_heads < 1 || d.q_len < 0 || d.kv_len < 1 ||
      d.head_dim < 1 || d.ld_probs < d.kv_len || d.q_heads % d.kv_heads != 0 ||
      !(std::isfinite(d.scale) && d.scale != 0.0f))
    return FOS_ERR_INVALID;
  if (in_dtype != FOS_BF16 && in_dtype != FOS_F16) return FOS_ERR_INVALID;
  if (out_dtype != FOS_F32 && out_dtype != FOS_BF16 && out_dtype != FOS_F16) return FOS_ERR_INVALID;
  if ((int64_t)d.batch * d.q_heads * d.q_len == 0) return FOS_OK;
  if (probs == nullptr || v == nullptr || out == nullptr) return FOS_ERR_INVALID;
  if (d.head_dim != 64 && d.head_dim != 128) return FOS_ERR_UNSUPPORTED;
  if (!aligned16(probs) || !aligned16(v) || !aligned16(out) || (d.ld_probs & 7) != 0)
    return FOS_ERR_UNSUPPORTED;
  if ((int64_t)d.batch * d.q_heads > 65535) return FOS_ERR_UNSUPPORTED;
  DevInfo *dev = nullptr;
  fos_status st = device_info(&dev);
  if (st != FOS_OK) return st;
  if ((st = bind_context(*dev)) != FOS_OK) return st;
  return run_pv(desc, in_dtype, out_dtype, probs, v, out, stream, dev->err, dev->max_smem);
}

extern "C" fos_status fos_grad_kv(const fos_pv_desc *desc, fos_dtype in_dtype,
                                  fos_dtype out_dtype, const void *a, const void *m, void *out,
                                  cudaStream_t stream) {
  if (desc == nullptr) return FOS_ERR_INVALID;
  const fos_pv_desc &d = *desc;
  if (d.batch < 0 || d.q_heads < 0 || d.kv_heads < 1 || d.q_len < 0 || d.kv_len < 0 ||
      d.head_dim < 1 || d.ld_probs < d.kv_len || d.q_heads % d.kv_heads != 0 || d.q_heads < 1 ||
      !(std::isfinite(d.scale) && d.scale != 0.0f))
    return FOS_ERR_INVALID;
  if (in_dtype != FOS_BF16 && in_dtype != FOS_F16) return FOS_ERR_INVALID;
  if (out_dtype != FOS_F32 && out_dtype != FOS_BF16 && out_dtype != FOS_F16) return FOS_ERR_INVALID;
  const int64_t nout = (int64_t)d.batch * d.kv_heads * d.kv_len * d.head_dim;
  if (nout == 0) return FOS_OK;
  if (out == nullptr) return FOS_ERR_INVALID;
  if (d.head_dim != 64 && d.head_dim != 128) return FOS_ERR_UNSUPPORTED;
  if (d.q_len == 0)  // a sum over no query position: every output is +0
    return cudaMemsetAsync(out, 0, (size_t)nout * dtype_size(out_dtype), stream) == cudaSuccess
               ? FOS_OK
               : FOS_ERR_CUDA;
  if (a == nullptr || m == nullptr) return FOS_ERR_INVALID;
  if (!aligned16(a) || !aligned16(m) || !aligned16(out) || (d.ld_probs & 7) != 0)
    return FOS_ERR_UNSUPPORTED;
  if ((int64_t)d.batch * d.kv_heads > 65535) return FOS_ERR_UNSUPPORTED;
  DevInfo *dev = nullptr;
  fos_status st = device_info(&dev);
  if (st != FOS_OK) return st;
  if ((st = bind_context(*dev)) != FOS_OK) return st;
  return run_kvgrad(desc, in_dtype, out_dtype, a, m, out, stream, dev->err, dev->max_smem);
}

extern "C" fos_status fos_sink_grad(const fos_desc *desc, const float *lse, const float *delta,
                                    float *d_sink, cudaStream_t stream,
                                    const fos_launch *launch) {
  fos_status st = check_desc(desc);
  if (st != FOS_OK) return st;
  if ((st = check_launch(launch)) != FOS_OK) return st;
  if (desc->sink == nullptr || lse == nullptr || delta == nullptr || d_sink == nullptr)
    return FOS_ERR_INVALID;
  if (desc->heads == 0) return FOS_OK;
  if (desc->rows == 0) return FOS_ERR_INVALID;  // heads > 0 with no rows: nothing defines d_sink
  return run_sink(desc, lse, delta, d_sink, stream, launch);
}

extern "C" fos_status fos_sink_grad_partials(const fos_desc *desc, int32_t batch_begin,
                                             int32_t batch_end, const float *lse,
                                             const float *delta, float *partials,
                                             cudaStream_t stream, const fos_launch *launch) {
  fos_status st = check_desc(desc);
  if (st != FOS_OK) return st;
  if ((st = check_launch(launch)) != FOS_OK) return st;
  if (desc->sink == nullptr || lse == nullptr || delta == nullptr || partials == nullptr)
    return FOS_ERR_INVALID;
  if (batch_begin < 0 || batch_end < batch_begin || batch_end > desc->batch)
    return FOS_ERR_INVALID;
  if (batch_end == batch_begin) return FOS_OK;  // an empty shard has no chunks
  // the shard's positions [b0 * q_len, b1 * q_len) of every head must be whole chunks of the
  // 256-position grid, except for a partial last chunk at the end of the batch
  const int64_t p0 = (int64_t)batch_begin * desc->q_len, p1 = (int64_t)batch_end * desc->q_len;
  if (p0 % kTileK != 0 || (batch_end < desc->batch && p1 % kTileK != 0)) return FOS_ERR_INVALID;
  if (desc->heads == 0 || p1 == p0) return FOS_OK;
  DevInfo *dev = nullptr;
  if ((st = device_info(&dev)) != FOS_OK) return st;
  SinkArgs a{};
  fill_sink_args(desc, &a);
  a.lse = lse;
  a.delta = delta;
  const int warps = (launch && launch->warps_per_cta) ? launch->warps_per_cta : kDefaultWarps;
  if (sink_partials_launch(a, batch_begin, batch_end, partials, warps * 32, stream) !=
      cudaSuccess)
    return FOS_ERR_CUDA;
  return FOS_OK;
}

extern "C" fos_status fos_sink_grad_merge(int32_t heads, int64_t nchunks, const float *partials,
                                          float *d_sink) {
  if (heads < 0 || nchunks < 0) return FOS_ERR_INVALID;
  if (heads > 0 && (d_sink == nullptr || (nchunks > 0 && partials == nullptr)))
    return FOS_ERR_INVALID;
  for (int32_t h = 0; h < heads; ++h) {
    // float32 additions in chunk order from +0, as the device sum does
    float total = 0.0f;
    for (int64_t c = 0; c < nchunks; ++c) total = total + partials[(int64_t)h * nchunks + c];
    d_sink[h] = total;
  }
  return FOS_OK;
}

extern "C" fos_status fos_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FOS_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return FOS_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return FOS_ERR_CUDA;
    return v == 2u ? FOS_ERR_INDEX : FOS_ERR_TIMEOUT;  // 2: a debug-build index check
  }
  return FOS_OK;
}

extern "C" const char *fos_status_string(fos_status status) {
  switch (status) {
    case FOS_OK: return "FOS_OK";
    case FOS_ERR_INVALID: return "FOS_ERR_INVALID: invalid argument";
    case FOS_ERR_UNSUPPORTED: return "FOS_ERR_UNSUPPORTED: valid but not supported by the kernels";
    case FOS_ERR_CUDA: return "FOS_ERR_CUDA: CUDA launch or runtime error";
    case FOS_ERR_TIMEOUT: return "FOS_ERR_TIMEOUT: a bounded wait in a kernel ran out";
    case FOS_ERR_INDEX: return "FOS_ERR_INDEX: an index check of the debug build failed";
  }
  return "unknown fos_status";
}

extern "C" const char *fos_contract_fingerprint(void) {
  return "fos-softmax contract 1; sm_103a; TILE_K=256; lane l owns keys 8l..8l+7 of a tile, "
         "combined in ascending order; warp xor tree 16,8,4,2,1 for max and sums; "
         "online merge of tile states left to right from (sink,1) or (-inf,0), "
         "S=S*exp(Mprev-M)+s_t*exp(m_t-M), exp(a-b):=1 when a==b; "
         "exp(x)=ex2.approx.f32(rn(x*rn(log2 e))); P=rn(e_j*rn(exp(m_t-M)/S)); "
         "LSE=M+logf(S); delta: lane fma chain, xor tree, tiles left to right; "
         "dS=fma(P,rn(dP-delta),+0); d_sink: rows of a head in (b,i) order, chunks of 256 "
         "with the same lane/tree layout, chunks left to right; "
         "float32 intermediates, one rounding to the I/O dtype (RNE); no FMA contraction, "
         "no fast-math, no atomics, no split rows, no tensor cores";
}
