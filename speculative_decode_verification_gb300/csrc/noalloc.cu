// noalloc.cu - the routed-expert call for callers that may not allocate device
// memory.  Its scratch is a fixed array compiled into the library; nothing
// here calls cudaMalloc, cudaFree or an allocating library routine.
#include <mutex>

#include "internal.h"
#include "verify.h"

namespace {

// Scratch of the routed-expert kernels: SwiGLU rows [k, T+1, I] bf16, per-rank
// partial outputs [k, T+1, H] fp32, an error word and the work-scheduling
// words (item counters, per-SM arrival counters, per-unit counts).  Every GPU that loads the library holds it until the process
// exits.  All calls on one device share it.
constexpr size_t kScratchBytes = VERIFY_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_scratch on this device
  int num_sms = 0;
  int moe_ctas_per_sm = 0;
};

std::mutex g_mutex;
DeviceSetup g_dev[kMaxDevices];

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// Once per device, with that device current: resolve the array's device
// address (the host-side name g_scratch is only a stand-in), set the kernels'
// launch attributes and read the SM count.
verify_status setup_device(int dev, DeviceSetup** out) {
  if (dev < 0 || dev >= kMaxDevices) return VERIFY_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceSetup& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return VERIFY_ECUDA;
    int dense_ctas = 0, moe_ctas = 0, sms = 0;
    if (vk::q4_setup_kernels(&dense_ctas, &moe_ctas) != cudaSuccess) return VERIFY_ECUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return VERIFY_ECUDA;
    d.scratch = static_cast<unsigned char*>(p);
    d.num_sms = sms;
    d.moe_ctas_per_sm = moe_ctas;
    d.ready = true;
  }
  *out = &d;
  return VERIFY_OK;
}

bool device_memory(const void* p, size_t align) {
  if (!p || reinterpret_cast<uintptr_t>(p) % align) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// A tiled operand (q4_tile) of the given layout.
bool valid_q4(const verify_q4_weight* W, int layout) {
  return W && W->group_size == 64 && W->bits == 4 && W->layout == layout && W->k_in % 64 == 0 && W->k_in >= 64 &&
         W->n_out >= 1 && device_memory(W->packed, 16);
}


}  // namespace

extern "C" verify_status q4_gather_experts_k_noalloc(
    const verify_q4_experts* gate_up, const verify_q4_experts* down, const float* logits, int64_t logits_ld,
    int top_k, const uint16_t* x, int k, int32_t* idx_out, float* w_out, void* y, int dtype_out,
    const verify_q4_weight* shared_gate_up, const verify_q4_weight* shared_down, const float* shared_gate_logit,
    int32_t* device_error, struct CUstream_st* stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return VERIFY_ECUDA;
  DeviceSetup* d = nullptr;
  verify_status s = setup_device(dev, &d);
  if (s) return s;

  // ---- arguments (all checked before anything is enqueued); the shape rules
  // are those of q4_gather_experts_k, with k limited to one pass
  if (!gate_up || !down) return VERIFY_EINVAL;
  const int E = gate_up->n_experts;
  const char* why = "";
  if (int rule = vk::moe_shape_status(k, VERIFY_PASS_K, E, down->n_experts, top_k, gate_up->w.n_out,
                                      gate_up->w.k_in, down->w.n_out, down->w.k_in, &why))
    return (verify_status)rule;
  if (!valid_q4(&gate_up->w, VERIFY_Q4_TILED_GATE_UP) || !valid_q4(&down->w, VERIFY_Q4_TILED_DOWN)) return VERIFY_EINVAL;
  const int H = gate_up->w.k_in, I = gate_up->w.n_out / 2;
  if (logits_ld < E) return VERIFY_EINVAL;
  if (dtype_out != VERIFY_F32 && dtype_out != VERIFY_BF16 && dtype_out != VERIFY_F32_ADD) return VERIFY_EINVAL;
  if (!device_memory(logits, 4) || !device_memory(x, 16) || !device_memory(idx_out, 4) || !device_memory(w_out, 4) ||
      !device_memory(y, dtype_out == VERIFY_BF16 ? 2 : 4))
    return VERIFY_EINVAL;
  if (device_error && !device_memory(device_error, 4)) return VERIFY_EINVAL;
  const int n_shared = (shared_gate_up != nullptr) + (shared_down != nullptr) + (shared_gate_logit != nullptr);
  if (n_shared != 0 && n_shared != 3) return VERIFY_EINVAL;
  if (n_shared == 3) {
    if (!valid_q4(shared_gate_up, VERIFY_Q4_TILED_GATE_UP) || !valid_q4(shared_down, VERIFY_Q4_TILED_DOWN) ||
        !device_memory(shared_gate_logit, 4))
      return VERIFY_EINVAL;
    if (shared_gate_up->n_out != 2 * I || shared_gate_up->k_in != H || shared_down->n_out != H ||
        shared_down->k_in != I)
      return VERIFY_EINVAL;
  }
  // ---- carve the fixed scratch; reject what does not fit
  const int TS = top_k + (n_shared ? 1 : 0);
  const size_t hbuf_bytes = round256((size_t)k * TS * I * sizeof(uint16_t));
  const size_t part_bytes = round256((size_t)k * TS * H * sizeof(float));
  const size_t word_bytes = round256((size_t)(1 + vk::kMoeSchedWords) * sizeof(int));  // error word, scheduling words
  if (hbuf_bytes + part_bytes + word_bytes > kScratchBytes) return VERIFY_EUNSUPPORTED;
  unsigned char* base = d->scratch;
  int* err_word = reinterpret_cast<int*>(base + hbuf_bytes + part_bytes);

  vk::MoeArgs a{};
  a.logits = logits; a.logits_ld = logits_ld; a.shared_logit = n_shared ? shared_gate_logit : nullptr;
  a.x = x;
  a.gu_tiles = reinterpret_cast<const uint8_t*>(gate_up->w.packed);
  a.dn_tiles = reinterpret_cast<const uint8_t*>(down->w.packed);
  if (n_shared) {
    a.sgu_tiles = reinterpret_cast<const uint8_t*>(shared_gate_up->packed);
    a.sdn_tiles = reinterpret_cast<const uint8_t*>(shared_down->packed);
  }
  a.gu_rt_bytes = vk::tile_row_bytes(H, vk::kExpertGroups);
  a.dn_rt_bytes = vk::tile_row_bytes(I, vk::kExpertGroups);
  a.hbuf = reinterpret_cast<uint16_t*>(base);
  a.part = reinterpret_cast<float*>(base + hbuf_bytes);
  a.work = err_word + 1;
  a.done = a.work + 2 + vk::kMoeSmSlots;
  a.idx_out = idx_out; a.w_out = w_out; a.y = y;
  a.err = device_error ? device_error : err_word;
  a.E = E; a.T = top_k; a.H = H; a.I = I; a.k = k; a.dtype = dtype_out;
  a.has_shared = n_shared ? 1 : 0;
  a.G = vk::moe_ctas_per_sm_for(k, top_k, E, a.has_shared, I, d->num_sms, d->moe_ctas_per_sm) * d->num_sms;
  a.n_sm = d->num_sms;
  // The error word and the scheduling words must start at zero: a previous
  // call may have stopped on a device error and left them set.
  if (cudaMemsetAsync(err_word, 0, (size_t)(1 + vk::kMoeSchedWords) * sizeof(int), stream) != cudaSuccess)
    return VERIFY_ECUDA;
  int launched = 0;
  if (vk::launch_moe(a, false, stream, &launched) != cudaSuccess) return VERIFY_ECUDA;
  return VERIFY_OK;
}
