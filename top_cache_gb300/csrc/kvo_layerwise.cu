// Layerwise prefill offload: "Layerwise and Sparse KV Cache Offloading
// Design", section 3 ("Buffer planning", "Execution pipeline", "Reuse
// invariant"), and the FlashOffloading explainer's prefill paragraph (four
// trays, tray B0 bound to the first layer, onload_layer_map lookahead).
//
// The path is made of layer-sized contiguous transfers, so it runs on the copy
// engines: loads on one library stream, saves on another, and the SMs stay with
// the caller's compute.  CUDA events carry every ordering:
//   load of layer l into buffer b   waits for the save of b's previous layer
//                                   (the reuse invariant, tracked per buffer);
//   compute of layer l              waits for that load (kvo_lw_layer);
//   save of layer l                 waits for that compute (kvo_lw_layer_done);
//   end of the pass                 waits for every save (kvo_lw_end).
// A buffer that still holds a layer's rows 0..L-1 (an independent layer, or a
// shared buffer that no other layer used since) is not reloaded.
#include <cstring>
#include <vector>

#include "kvo_internal.cuh"

struct kvo_lw {
  kvo_lw_config cfg{};
  int n_phys = 0;
  std::vector<int32_t> phys;         // buffer of each layer
  std::vector<int32_t> prev_same;    // previous layer of the same buffer, or -1
  uint16_t* host = nullptr;          // pinned pool [N][max_tokens][row]
  size_t host_map_bytes = 0, host_huge = 0;
  uint16_t* buf = nullptr;           // device buffers [n_phys][max_tokens][row]
  cudaStream_t load_s = nullptr, save_s = nullptr;
  std::vector<cudaEvent_t> ev_load;  // per layer: its buffer holds rows 0..L-1
  std::vector<cudaEvent_t> ev_comp;  // per layer: the caller's compute is done
  std::vector<cudaEvent_t> ev_saved; // per buffer: the save of its last layer is done
  std::vector<char> saved_rec;       // per buffer: ev_saved has been recorded
  std::vector<int32_t> holds;        // per buffer: the layer whose rows it holds, or -1
  std::vector<int64_t> holds_len;    // per buffer: how many of that layer's rows
  cudaEvent_t ev_begin = nullptr, ev_end = nullptr;
  int64_t length = 0, chunk = 0;
  bool in_pass = false;
  int next_layer = 0, next_load = 0, load_target = -1;
  uint64_t bytes_h2d = 0, bytes_d2h = 0;
};

namespace {

size_t row_bytes(const kvo_lw* lw) { return (size_t)lw->cfg.row_elems * 2; }
uint16_t* host_layer(const kvo_lw* lw, int l) {
  return lw->host + (size_t)l * (size_t)lw->cfg.max_tokens * lw->cfg.row_elems;
}
uint16_t* dev_buffer(const kvo_lw* lw, int b) {
  return lw->buf + (size_t)b * (size_t)lw->cfg.max_tokens * lw->cfg.row_elems;
}

struct Guard {
  int prev = -1;
  explicit Guard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~Guard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

void release(kvo_lw* lw) {
  for (auto e : lw->ev_load) if (e) cudaEventDestroy(e);
  for (auto e : lw->ev_comp) if (e) cudaEventDestroy(e);
  for (auto e : lw->ev_saved) if (e) cudaEventDestroy(e);
  if (lw->ev_begin) cudaEventDestroy(lw->ev_begin);
  if (lw->ev_end) cudaEventDestroy(lw->ev_end);
  if (lw->load_s) cudaStreamDestroy(lw->load_s);
  if (lw->save_s) cudaStreamDestroy(lw->save_s);
  if (lw->buf) cudaFree(lw->buf);
  kvo::free_pinned(lw->host, lw->host_map_bytes);
  delete lw;
}

// Issue the loads of layers next_load..load_target (in order) on the load
// stream.  A load into a buffer whose previous layer in this pass has not been
// saved yet (its kvo_lw_layer_done not called) waits on the host side: it is
// issued from that kvo_lw_layer_done.  A layer's own load is never held back
// when its compute begins, because that previous layer comes before it.
cudaError_t issue_loads(kvo_lw* lw) {
  const int N = lw->cfg.n_layers;
  const int upto = lw->load_target < N - 1 ? lw->load_target : N - 1;
  cudaError_t e = cudaSuccess;
  for (; lw->next_load <= upto && e == cudaSuccess; ++lw->next_load) {
    const int l = lw->next_load, b = lw->phys[(size_t)l];
    const bool resident = lw->holds[(size_t)b] == l && lw->holds_len[(size_t)b] >= lw->length;
    if (!resident) {
      const int prev = lw->prev_same[(size_t)l];
      if (prev >= 0 && prev >= lw->next_layer) break;  // its save is not enqueued yet
      // reuse invariant: the buffer's previous layer has been saved
      if (lw->saved_rec[(size_t)b]) e = cudaStreamWaitEvent(lw->load_s, lw->ev_saved[(size_t)b], 0);
      if (e == cudaSuccess && lw->length > 0) {
        const size_t bytes = (size_t)lw->length * row_bytes(lw);
        e = cudaMemcpyAsync(dev_buffer(lw, b), host_layer(lw, l), bytes, cudaMemcpyHostToDevice, lw->load_s);
        lw->bytes_h2d += bytes;
      }
      lw->holds[(size_t)b] = l;
      lw->holds_len[(size_t)b] = lw->length;
    }
    if (e == cudaSuccess) e = cudaEventRecord(lw->ev_load[(size_t)l], lw->load_s);
  }
  return e;
}

}  // namespace

extern "C" {

int kvo_lw_create(const kvo_lw_config* cfg, kvo_lw** out) {
  if (!out) return kvo::set_error(KVO_EINVAL, "out is NULL");
  *out = nullptr;
  if (!cfg) return kvo::set_error(KVO_EINVAL, "cfg is NULL");
  const kvo_lw_config c = *cfg;
  if (c.n_layers < 1 || c.n_layers > 4096) return kvo::set_error(KVO_EINVAL, "n_layers out of range");
  if (c.n_independent < 0 || c.n_independent > c.n_layers) return kvo::set_error(KVO_EINVAL, "n_independent out of range");
  if (c.n_shared < 0 || (c.n_independent < c.n_layers && c.n_shared < 1))
    return kvo::set_error(KVO_EINVAL, "reusable layers need at least one shared buffer");
  if (c.lookahead < 1) return kvo::set_error(KVO_EINVAL, "lookahead must be >= 1");
  if (c.max_tokens < 1) return kvo::set_error(KVO_EINVAL, "max_tokens must be >= 1");
  if (c.row_elems < 8 || (c.row_elems * 2) % 16 != 0) return kvo::set_error(KVO_EINVAL, "row bytes must be a multiple of 16");
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || c.device < 0 || c.device >= ndev)
    return kvo::set_error(KVO_EINVAL, "no such device");
  Guard g(c.device);
  kvo_lw* lw = new kvo_lw();
  lw->cfg = c;
  // plan (reading R14 of the oracle)
  const int N = c.n_layers, I = c.n_independent, R = N - I;
  const int S = R > 0 ? (c.n_shared < R ? c.n_shared : R) : 0;
  lw->n_phys = I + S;
  lw->phys.resize((size_t)N);
  for (int l = 0; l < I; ++l) lw->phys[(size_t)l] = l;
  for (int k = 0; k < R; ++k) lw->phys[(size_t)(I + k)] = I + k % S;
  lw->prev_same.assign((size_t)N, -1);
  {
    std::vector<int32_t> last((size_t)(I + S), -1);
    for (int l = 0; l < N; ++l) {
      lw->prev_same[(size_t)l] = last[(size_t)lw->phys[(size_t)l]];
      last[(size_t)lw->phys[(size_t)l]] = l;
    }
  }
  const size_t per = (size_t)c.max_tokens * (size_t)c.row_elems * 2;
  cudaError_t e = kvo::alloc_pinned(per * (size_t)N, reinterpret_cast<void**>(&lw->host), &lw->host_map_bytes, &lw->host_huge);
  if (e == cudaSuccess) memset(lw->host, 0, per * (size_t)N);
  if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&lw->buf), per * (size_t)lw->n_phys);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&lw->load_s, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&lw->save_s, cudaStreamNonBlocking);
  lw->ev_load.assign((size_t)N, nullptr);
  lw->ev_comp.assign((size_t)N, nullptr);
  lw->ev_saved.assign((size_t)lw->n_phys, nullptr);
  lw->saved_rec.assign((size_t)lw->n_phys, 0);
  lw->holds.assign((size_t)lw->n_phys, -1);
  lw->holds_len.assign((size_t)lw->n_phys, 0);
  for (int l = 0; l < N && e == cudaSuccess; ++l) {
    e = cudaEventCreateWithFlags(&lw->ev_load[(size_t)l], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&lw->ev_comp[(size_t)l], cudaEventDisableTiming);
  }
  for (int b = 0; b < lw->n_phys && e == cudaSuccess; ++b)
    e = cudaEventCreateWithFlags(&lw->ev_saved[(size_t)b], cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&lw->ev_begin, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&lw->ev_end, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    release(lw);
    cudaGetLastError();  // a failed allocation is not left as the thread's last CUDA error
    return e == cudaErrorMemoryAllocation ? kvo::set_error(KVO_ENOMEM, "layerwise buffers")
                                          : kvo::set_cuda_error(e, "layerwise create");
  }
  *out = lw;
  return KVO_OK;
}

int kvo_lw_destroy(kvo_lw* lw) {
  if (!lw) return KVO_OK;
  Guard g(lw->cfg.device);
  cudaStreamSynchronize(lw->load_s);
  cudaStreamSynchronize(lw->save_s);
  release(lw);
  return KVO_OK;
}

int kvo_lw_plan(kvo_lw* lw, int32_t* n_phys, int32_t* phys_of_layer) {
  if (!lw || !n_phys) return kvo::set_error(KVO_EINVAL, "NULL argument");
  *n_phys = lw->n_phys;
  if (phys_of_layer) memcpy(phys_of_layer, lw->phys.data(), lw->phys.size() * 4);
  return KVO_OK;
}

void* kvo_lw_host_rows(kvo_lw* lw, int32_t layer) {
  if (!lw || layer < 0 || layer >= lw->cfg.n_layers) {
    kvo::set_error(KVO_EINVAL, "bad layer");
    return nullptr;
  }
  return host_layer(lw, layer);
}

int kvo_lw_set_length(kvo_lw* lw, int64_t tokens) {
  if (!lw) return kvo::set_error(KVO_EINVAL, "handle is NULL");
  if (lw->in_pass) return kvo::set_error(KVO_EINVAL, "inside a pass");
  if (tokens < 0 || tokens > lw->cfg.max_tokens) return kvo::set_error(KVO_ERANGE, "length out of range");
  Guard g(lw->cfg.device);
  cudaError_t e = cudaStreamSynchronize(lw->load_s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(lw->save_s);
  if (e != cudaSuccess) return kvo::set_cuda_error(e, "layerwise streams");
  lw->length = tokens;
  for (auto& h : lw->holds) h = -1;
  return KVO_OK;
}

int kvo_lw_begin(kvo_lw* lw, int64_t chunk_tokens, void* stream) {
  if (!lw) return kvo::set_error(KVO_EINVAL, "handle is NULL");
  if (lw->in_pass) return kvo::set_error(KVO_EINVAL, "a pass is already open");
  if (chunk_tokens < 0 || lw->length + chunk_tokens > lw->cfg.max_tokens)
    return kvo::set_error(KVO_ERANGE, "length + chunk past max_tokens");
  Guard g(lw->cfg.device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaEventRecord(lw->ev_begin, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(lw->load_s, lw->ev_begin, 0);
  if (e != cudaSuccess) return kvo::set_cuda_error(e, "layerwise begin");
  lw->chunk = chunk_tokens;
  lw->in_pass = true;
  lw->next_layer = 0;
  lw->next_load = 0;
  lw->load_target = lw->cfg.lookahead - 1;
  e = issue_loads(lw);
  if (e != cudaSuccess) return kvo::set_cuda_error(e, "layerwise loads");
  return KVO_OK;
}

int kvo_lw_layer(kvo_lw* lw, int32_t layer, void** buffer, void* stream) {
  if (!lw || !buffer) return kvo::set_error(KVO_EINVAL, "NULL argument");
  if (!lw->in_pass) return kvo::set_error(KVO_EINVAL, "no open pass");
  if (layer != lw->next_layer) return kvo::set_error(KVO_EINVAL, "layers must come in order");
  Guard g(lw->cfg.device);
  if (layer + lw->cfg.lookahead > lw->load_target) lw->load_target = layer + lw->cfg.lookahead;
  cudaError_t e = issue_loads(lw);
  if (e == cudaSuccess && lw->next_load <= layer) e = cudaErrorNotReady;  // cannot happen: see issue_loads
  if (e == cudaSuccess) e = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), lw->ev_load[(size_t)layer], 0);
  if (e != cudaSuccess) return kvo::set_cuda_error(e, "layerwise layer");
  *buffer = dev_buffer(lw, lw->phys[(size_t)layer]);
  return KVO_OK;
}

int kvo_lw_layer_done(kvo_lw* lw, int32_t layer, void* stream) {
  if (!lw) return kvo::set_error(KVO_EINVAL, "handle is NULL");
  if (!lw->in_pass || layer != lw->next_layer) return kvo::set_error(KVO_EINVAL, "layer is not the open one");
  Guard g(lw->cfg.device);
  const int b = lw->phys[(size_t)layer];
  cudaError_t e = cudaEventRecord(lw->ev_comp[(size_t)layer], static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamWaitEvent(lw->save_s, lw->ev_comp[(size_t)layer], 0);
  if (e == cudaSuccess && lw->chunk > 0) {
    const size_t off = (size_t)lw->length * lw->cfg.row_elems, bytes = (size_t)lw->chunk * row_bytes(lw);
    e = cudaMemcpyAsync(host_layer(lw, layer) + off, dev_buffer(lw, b) + off, bytes, cudaMemcpyDeviceToHost, lw->save_s);
    lw->bytes_d2h += bytes;
  }
  if (e == cudaSuccess) e = cudaEventRecord(lw->ev_saved[(size_t)b], lw->save_s);
  if (e != cudaSuccess) return kvo::set_cuda_error(e, "layerwise save");
  lw->saved_rec[(size_t)b] = 1;
  lw->holds_len[(size_t)b] = lw->length + lw->chunk;  // the buffer now holds the chunk too
  ++lw->next_layer;
  e = issue_loads(lw);  // loads that waited for this save
  if (e != cudaSuccess) return kvo::set_cuda_error(e, "layerwise loads");
  return KVO_OK;
}

int kvo_lw_end(kvo_lw* lw, void* stream) {
  if (!lw) return kvo::set_error(KVO_EINVAL, "handle is NULL");
  if (!lw->in_pass || lw->next_layer != lw->cfg.n_layers) return kvo::set_error(KVO_EINVAL, "pass not complete");
  Guard g(lw->cfg.device);
  cudaError_t e = cudaEventRecord(lw->ev_end, lw->save_s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), lw->ev_end, 0);
  if (e != cudaSuccess) return kvo::set_cuda_error(e, "layerwise end");
  lw->length += lw->chunk;
  lw->chunk = 0;
  lw->in_pass = false;
  return KVO_OK;
}

int kvo_lw_stats(kvo_lw* lw, uint64_t* bytes_h2d, uint64_t* bytes_d2h) {
  if (!lw || !bytes_h2d || !bytes_d2h) return kvo::set_error(KVO_EINVAL, "NULL argument");
  *bytes_h2d = lw->bytes_h2d;
  *bytes_d2h = lw->bytes_d2h;
  return KVO_OK;
}

}  // extern "C"
