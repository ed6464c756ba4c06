// h3q_host_pipeline.cu -- the grouped W8A8 Linear from and to pinned host
// memory: X goes up, the G outputs come down, in row chunks that overlap the
// two copy directions with the grouped calls (A2 + A3 + A4 per chunk).
//
// Three streams carry it: uploads, the grouped calls, downloads.  Chunk c's
// call waits for its upload; its downloads wait for the call.  The host link
// is the bound (the outputs are G times the input), so the schedule aims to
// keep the download direction busy from as early as possible: the first
// chunks are small (the first download starts after a short call) and grow to
// the steady chunk size.  Every chunk's rows are its own regions of the device
// staging buffers, so no chunk waits for another's copies; the workspace is
// reused chunk after chunk on the call stream, which orders it.
#include <map>
#include <mutex>
#include <vector>

#include "h3q_abi_checks.cuh"
#include "h3q_internal.cuh"

namespace {

constexpr int64_t kRowQuantum = 16;  // chunk boundaries: keep every row block 16-byte aligned
constexpr int64_t kRampChunks = 32;  // bound on the chunks before the steady size

// Row ranges of the chunks: first_rows, doubling, up to chunk_rows, then
// chunk_rows until M is covered (the last one takes what is left).
std::vector<std::pair<int64_t, int64_t>> chunk_plan(int64_t M, int64_t chunk_rows,
                                                    int64_t first_rows) {
  std::vector<std::pair<int64_t, int64_t>> plan;
  int64_t rows = first_rows;
  for (int64_t r0 = 0; r0 < M;) {
    const int64_t r1 = r0 + rows < M ? r0 + rows : M;
    plan.emplace_back(r0, r1);
    r0 = r1;
    rows = rows * 2 < chunk_rows ? rows * 2 : chunk_rows;
  }
  return plan;
}

int64_t default_first_rows(int64_t chunk_rows) {
  const int64_t q = (chunk_rows / 4 + kRowQuantum - 1) / kRowQuantum * kRowQuantum;
  return q < kRowQuantum ? kRowQuantum : q;
}

// Upper bound on the chunks of any plan for (M, chunk_rows): the ramp has
// fewer than kRampChunks entries (it doubles from >= 16 rows), and after it
// every chunk but the last is full.
int64_t max_chunks(int64_t M, int64_t chunk_rows) {
  return (M + chunk_rows - 1) / chunk_rows + kRampChunks;
}

size_t round256(size_t b) { return (b + 255u) & ~size_t(255); }

// Events are created once per device and reused call after call: the call
// synchronises before it returns, so no event of a finished call is pending,
// and the lock keeps two host threads from sharing them.
struct EventPool {
  std::mutex m;
  std::vector<cudaEvent_t> ev;
};

EventPool& event_pool(int dev) {
  static std::mutex pools_m;
  static std::map<int, EventPool*> pools;
  std::lock_guard<std::mutex> lock(pools_m);
  EventPool*& p = pools[dev];
  if (!p) p = new EventPool;
  return *p;
}

bool pinned_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

}  // namespace

extern "C" {

size_t h3q_linear_w8a8_grouped_host_workspace_bytes(int G, int64_t M, int64_t N, int64_t K,
                                                    int64_t chunk_rows) {
  if (G < 1 || G > h3q::kMaxGroup || M < 1 || N < 1 || K < 1) return 0;
  if (chunk_rows < kRowQuantum || chunk_rows % kRowQuantum) return 0;
  const int64_t rows = chunk_rows < M ? chunk_rows : M;
  return round256(h3q::workspace_layout(rows, N, K, G).total) +
         round256(size_t(max_chunks(M, chunk_rows)) * sizeof(uint32_t));
}

int64_t h3q_linear_w8a8_grouped_host_chunks(int64_t M, int64_t chunk_rows, int64_t first_rows,
                                            int64_t* rows_out, int64_t capacity) {
  if (M < 1 || chunk_rows < kRowQuantum || chunk_rows % kRowQuantum) return -1;
  if (first_rows == 0) first_rows = default_first_rows(chunk_rows);
  if (first_rows < kRowQuantum || first_rows % kRowQuantum || first_rows > chunk_rows) return -1;
  const std::vector<std::pair<int64_t, int64_t>> plan = chunk_plan(M, chunk_rows, first_rows);
  for (size_t c = 0; rows_out && c < plan.size() && int64_t(c) < capacity; ++c)
    rows_out[c] = plan[c].second - plan[c].first;
  return int64_t(plan.size());
}

h3q_status h3q_linear_w8a8_grouped_host(const uint16_t* x_host, int G, const int8_t* const* wq,
                                        const float* const* ws, const uint16_t* const* bias,
                                        int64_t M, int64_t N, int64_t K,
                                        uint16_t* const* y_host, uint16_t* x_dev, float* xs,
                                        uint16_t* const* y_dev, int64_t chunk_rows,
                                        int64_t first_rows, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream,
                                        cudaStream_t h2d_stream, cudaStream_t d2h_stream) {
  if (G < 1 || G > h3q::kMaxGroup) return H3Q_ERR_INVALID_ARG;
  if (!x_host || !wq || !ws || !y_host || !x_dev || !xs || !y_dev || !workspace)
    return H3Q_ERR_INVALID_ARG;
  for (int g = 0; g < G; ++g)
    if (!wq[g] || !ws[g] || !y_host[g] || !y_dev[g]) return H3Q_ERR_INVALID_ARG;
  if (h3q_status st = h3q::check_shape(M, N, K)) return st;
  if (chunk_rows < kRowQuantum || chunk_rows % kRowQuantum) return H3Q_ERR_INVALID_ARG;
  if (first_rows == 0) first_rows = default_first_rows(chunk_rows);
  if (first_rows < kRowQuantum || first_rows % kRowQuantum || first_rows > chunk_rows)
    return H3Q_ERR_INVALID_ARG;
  if (workspace_bytes < h3q_linear_w8a8_grouped_host_workspace_bytes(G, M, N, K, chunk_rows))
    return H3Q_ERR_INVALID_ARG;
  if (!h3q::aligned16(x_host) || !h3q::aligned16(x_dev) || !h3q::aligned16(xs) ||
      !h3q::aligned16(workspace))
    return H3Q_ERR_MISALIGNED;
  for (int g = 0; g < G; ++g)
    if (!h3q::aligned16(y_host[g]) || !h3q::aligned16(y_dev[g])) return H3Q_ERR_MISALIGNED;
  if (h3q_status st = h3q::check_device()) return st;
  // Pageable host memory would make every copy synchronous: the pipeline needs
  // page-locked buffers.
  if (!pinned_host(x_host)) return H3Q_ERR_INVALID_ARG;
  for (int g = 0; g < G; ++g)
    if (!pinned_host(y_host[g])) return H3Q_ERR_INVALID_ARG;

  const std::vector<std::pair<int64_t, int64_t>> plan = chunk_plan(M, chunk_rows, first_rows);
  const int64_t rows_ws = chunk_rows < M ? chunk_rows : M;
  const size_t call_bytes = round256(h3q::workspace_layout(rows_ws, N, K, G).total);
  uint8_t* wsp = static_cast<uint8_t*>(workspace);
  uint32_t* slots = reinterpret_cast<uint32_t*>(wsp + call_bytes);
  const size_t nchunks = plan.size();

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return H3Q_ERR_CUDA;
  EventPool& pool = event_pool(dev);
  std::lock_guard<std::mutex> lock(pool.m);
  const size_t nev = 3 + 2 * nchunks;  // fork, two joins, per chunk: uploaded, computed
  while (pool.ev.size() < nev) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return H3Q_ERR_CUDA;
    pool.ev.push_back(e);
  }
  cudaEvent_t ev_fork = pool.ev[0], ev_h2d_done = pool.ev[1], ev_d2h_done = pool.ev[2];
  auto ev_in = [&](size_t c) { return pool.ev[3 + 2 * c]; };
  auto ev_out = [&](size_t c) { return pool.ev[4 + 2 * c]; };

  // The copy streams start after whatever the caller queued on `stream`.
  h3q_status st = H3Q_OK;
  if (cudaEventRecord(ev_fork, stream) != cudaSuccess ||
      cudaStreamWaitEvent(h2d_stream, ev_fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(d2h_stream, ev_fork, 0) != cudaSuccess)
    return H3Q_ERR_CUDA;

  // The G outputs as one [G, M, N] buffer on each side: a chunk's G
  // downloads are one 2D copy (fewer, larger copies run faster).  Outputs
  // that only happen to lie back to back in separate allocations may be
  // refused as one copy; then the copies go one by one.
  bool even = G > 1;
  for (int g = 1; even && g < G; ++g)
    even = y_host[g] - y_host[g - 1] == M * N && y_dev[g] - y_dev[g - 1] == M * N;

  size_t done = 0;  // chunks fully enqueued
  for (size_t c = 0; c < nchunks && st == H3Q_OK; ++c) {
    const int64_t r0 = plan[c].first, rows = plan[c].second - plan[c].first;
    if (cudaMemcpyAsync(x_dev + r0 * K, x_host + r0 * K, size_t(rows * K) * 2u,
                        cudaMemcpyHostToDevice, h2d_stream) != cudaSuccess ||
        cudaEventRecord(ev_in(c), h2d_stream) != cudaSuccess ||
        cudaStreamWaitEvent(stream, ev_in(c), 0) != cudaSuccess) {
      st = H3Q_ERR_CUDA;
      break;
    }
    uint16_t* yc[h3q::kMaxGroup];
    for (int g = 0; g < G; ++g) yc[g] = y_dev[g] + r0 * N;
    st = h3q_linear_w8a8_grouped(x_dev + r0 * K, nullptr, xs + r0, G, wq, ws, bias, rows, N, K,
                                 yc, workspace, call_bytes, stream);
    if (st != H3Q_OK) break;
    // This chunk's error word, kept: the next chunk's call clears the status block.
    const uint8_t* word = wsp + h3q::workspace_layout(rows, 1, K).status;
    if (cudaMemcpyAsync(slots + c, word, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream) !=
            cudaSuccess ||
        cudaEventRecord(ev_out(c), stream) != cudaSuccess ||
        cudaStreamWaitEvent(d2h_stream, ev_out(c), 0) != cudaSuccess) {
      st = H3Q_ERR_CUDA;
      break;
    }
    if (even) {
      // the chunk's rows of all G outputs in one copy
      const size_t pitch = size_t(M * N) * 2u;
      if (cudaMemcpy2DAsync(y_host[0] + r0 * N, pitch, y_dev[0] + r0 * N, pitch,
                            size_t(rows * N) * 2u, size_t(G), cudaMemcpyDeviceToHost,
                            d2h_stream) != cudaSuccess) {
        cudaGetLastError();   // refused at the call, nothing enqueued
        even = false;
      }
    }
    if (!even) {
      for (int g = 0; g < G && st == H3Q_OK; ++g)
        if (cudaMemcpyAsync(y_host[g] + r0 * N, y_dev[g] + r0 * N, size_t(rows * N) * 2u,
                            cudaMemcpyDeviceToHost, d2h_stream) != cudaSuccess)
          st = H3Q_ERR_CUDA;
    }
    if (st == H3Q_OK) ++done;
  }
  // Join both copy streams into `stream` and wait for everything enqueued,
  // whether or not every chunk was: no copy may still be running at return.
  const bool joined = cudaEventRecord(ev_h2d_done, h2d_stream) == cudaSuccess &&
                      cudaEventRecord(ev_d2h_done, d2h_stream) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, ev_h2d_done, 0) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, ev_d2h_done, 0) == cudaSuccess;
  std::vector<uint32_t> words(done);
  if (joined && done &&
      cudaMemcpyAsync(words.data(), slots, done * sizeof(uint32_t), cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess)
    st = st == H3Q_OK ? H3Q_ERR_CUDA : st;
  const cudaError_t sync = joined ? cudaStreamSynchronize(stream) : cudaDeviceSynchronize();
  if (st != H3Q_OK) return st;
  if (!joined || sync != cudaSuccess) return h3q::from_cuda(joined ? sync : cudaErrorUnknown);
  for (uint32_t w : words)
    if (w) return H3Q_ERR_TIMEOUT;
  return H3Q_OK;
}

}  // extern "C"
