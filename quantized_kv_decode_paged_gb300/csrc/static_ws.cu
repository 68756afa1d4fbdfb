// static_ws.cu — decode_attn_paged_static_ws: the split-KV paged decode with
// its scratch taken from a buffer compiled into the library, for callers
// that must not allocate device memory themselves.
//
// Who needs it: code that runs where cudaMalloc is not an option — an
// inference-server plugin whose host framework owns all device memory, a
// process held to a fixed device-memory budget, or a latency-critical loop
// that cannot afford cudaMalloc's implicit device synchronisation.
//
// The buffer is a file-scope __device__ array of DECODE_ATTN_STATIC_WS_BYTES
// bytes; every GPU that loads this library holds it until the process exits.
// Host code cannot pass the array's name to a kernel (on the host it is only
// a stand-in symbol), so the first call on each device looks up its device
// address with cudaGetSymbolAddress, with that device current, and keeps it.
// The address is kept together with the unique id of the
// context it was looked up in: after cudaDeviceReset the device gets a new
// context, and the next call looks the address up again (that call is then
// a first call).
//
// Every call uses the same array.  The ticket counters at its start must be
// zero when a call begins; each call clears them on its stream before the
// launch.  Calls whose work overlaps on the GPU (different streams without
// ordering, or several host threads) race on the array.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/decode_attn.h"
#include "launch.h"

namespace {

constexpr size_t kStaticWsBytes = DECODE_ATTN_STATIC_WS_BYTES;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the current context (never reused within a process), or 0.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

constexpr int kMaxDevices = 128;
struct CachedAddress {
  unsigned long long ctx_id;
  void* ptr;
};
CachedAddress g_ws_addr[kMaxDevices] = {};
std::mutex g_ws_mu;

// Device address of g_static_ws on the current device, looked up once per
// device and context.
int static_ws_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DA_ERR_UNSUPPORTED;
  // With no context yet (the first runtime call on this device), the id is
  // 0; the symbol lookup then creates the context and the id is read again.
  unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_ws_mu);
  CachedAddress& c = g_ws_addr[dev];
  if (id == 0 || !c.ptr || c.ctx_id != id) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || !ptr) return DA_ERR_CUDA;
    id = current_context_id();
    if (id == 0) return DA_ERR_CUDA;
    c.ptr = ptr;
    c.ctx_id = id;
  }
  *out = c.ptr;
  return DA_OK;
}

}  // namespace

extern "C" int decode_attn_paged_static_ws(const da_params* p, const float* q,
                                           const uint16_t* k_pool, const uint16_t* v_pool,
                                           const int32_t* block_table, const int32_t* seq_lens,
                                           const int32_t* q_pos, float* out, float* lse,
                                           int32_t* dev_status, void* stream) {
  if (!p) return DA_ERR_INVALID;
  const size_t need = decode_attn_workspace_size(p);
  if (need == 0) return DA_ERR_INVALID;
  if (need > kStaticWsBytes) return DA_ERR_WORKSPACE;
  const size_t tickets = da::workspace_ticket_bytes();
  if (tickets == 0 || tickets > need) return DA_ERR_CUDA;
  void* ws = nullptr;
  int st = static_ws_address(&ws);
  if (st != DA_OK) return st;
  if (cudaMemsetAsync(ws, 0, tickets, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DA_ERR_CUDA;
  return decode_attn_paged(p, q, k_pool, v_pool, block_table, seq_lens, q_pos, out, lse, ws, need,
                           dev_status, stream);
}
