// attn_static.cu -- split-K decode attention with its scratch in a static
// device array, for callers that cannot allocate device memory.
//
// nc_attn_decode keeps the split partials in a model's workspace, which
// nc_model_create allocates with cudaMalloc. Some callers cannot do that:
// code that runs while another thread of the process holds a stream in
// global-mode capture (cudaMalloc is not permitted then), code whose device
// memory belongs to a host framework's allocator that forbids raw cudaMalloc,
// and latency-critical loops that cannot pay cudaMalloc's implicit
// synchronisation. nc_attn_decode_static serves them: it needs no model and
// allocates nothing; the partials go to g_attn_scratch below.
//
// g_attn_scratch is a file-scope __device__ array, so every GPU that loads
// this library holds kStaticAttnScratchFloats * 4 bytes until the process
// exits. In host code its name is only a host-side stand-in, not a device
// address: passing it to a kernel would fault, or on a GPU that can reach
// host memory, silently use the wrong memory. The device address is taken
// with cudaGetSymbolAddress, with that device current: on the first call made
// on a device, and again on every call whose stream is not capturing (so a
// context created anew after a device reset is picked up); a capturing call
// uses the address looked up last.
//
// Errors the kernel finds on the device (an expired bounded wait, a block
// table entry or position that disagrees with the host copy) go to the static
// word g_attn_status, read and cleared by nc_attn_decode_static_status.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace nc {

// Partials of one call: [B][Hq][splits][D + 2] floats, at most 4 MiB.
constexpr size_t kStaticAttnScratchFloats = size_t(1) << 20;
static __device__ __align__(256) float g_attn_scratch[kStaticAttnScratchFloats];
// Merge tickets of one call, [B][Hkv]: zero at load, and the kernel leaves
// every ticket it used at zero again.
constexpr int kStaticAttnTickets = 1024;
static __device__ unsigned int g_attn_tickets[kStaticAttnTickets];
// Device-side error word of the calls (0 = none; else the first nc_status a
// kernel recorded since it was last read).
static __device__ int g_attn_status;

constexpr int kMaxDevices = 64;
static float* g_scratch_ptr[kMaxDevices];
static unsigned int* g_ticket_ptr[kMaxDevices];
static int* g_status_ptr[kMaxDevices];
static std::mutex g_scratch_mutex;

// Device addresses of g_attn_scratch, g_attn_tickets and g_attn_status on the
// current device: looked up on the first call on the device and on every
// call whose stream is not capturing; while capturing, the last lookup.
static cudaError_t static_scratch(cudaStream_t s, float** out, unsigned int** tickets,
                                  int** status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const bool capturing = cudaStreamIsCapturing(s, &cs) != cudaSuccess ||
                         cs != cudaStreamCaptureStatusNone;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr || !capturing) {
    void* p = nullptr;
    void* t = nullptr;
    void* w = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&t, g_attn_tickets);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&w, g_attn_status);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float*>(p);
    g_ticket_ptr[dev] = static_cast<unsigned int*>(t);
    g_status_ptr[dev] = static_cast<int*>(w);
  }
  *out = g_scratch_ptr[dev];
  *tickets = g_ticket_ptr[dev];
  *status = g_status_ptr[dev];
  return cudaSuccess;
}

}  // namespace nc

using namespace nc;

extern "C" nc_status nc_attn_decode_static(int n_q_heads, int n_kv_heads, int head_dim,
                                           int n_layers, int layer, int B, const float* q,
                                           const int32_t* positions_dev,
                                           const int32_t* positions_host,
                                           const nc_kv_cache* kv, float* out, void* stream) {
  NC_CHECK(q && positions_dev && positions_host && out && kv && kv->k && kv->v,
           NC_ERR_INVALID_ARGUMENT, "null pointer");
  NC_CHECK(head_dim == 64 || head_dim == 128, NC_ERR_SHAPE, "head_dim must be 64 or 128");
  NC_CHECK(n_q_heads > 0 && n_kv_heads > 0 && n_q_heads % n_kv_heads == 0 &&
               n_q_heads / n_kv_heads <= 8,
           NC_ERR_SHAPE, "n_q_heads must be a multiple of n_kv_heads, group at most 8");
  NC_CHECK(layer >= 0 && layer < n_layers, NC_ERR_SHAPE, "layer %d outside [0, %d)", layer,
           n_layers);
  NC_CHECK(B >= 1 && B <= 16, NC_ERR_CAPACITY, "batch %d outside [1, 16]", B);
  NC_CHECK(kv->dtype == NC_KV_F32 || kv->dtype == NC_KV_BF16, NC_ERR_DTYPE, "unknown kv dtype");
  NC_CHECK(reinterpret_cast<uintptr_t>(kv->k) % 16 == 0 && reinterpret_cast<uintptr_t>(kv->v) % 16 == 0,
           NC_ERR_INVALID_ARGUMENT, "kv cache pointers must be 16-byte aligned");
  int cap = 0;
  if (!kv->paged) {
    NC_CHECK(kv->batch_capacity >= B && kv->max_ctx >= 1, NC_ERR_CAPACITY,
             "contiguous cache smaller than the batch");
    cap = kv->max_ctx;
  } else {
    NC_CHECK(kv->block_table && kv->block_table_host && kv->block_size >= 1 &&
                 kv->num_blocks >= 1 && kv->max_blocks_per_seq >= 1,
             NC_ERR_INVALID_ARGUMENT, "paged cache needs block tables and positive sizes");
    cap = kv->max_blocks_per_seq * kv->block_size;
  }
  for (int b = 0; b < B; ++b) {
    const int p = positions_host[b];
    NC_CHECK(p >= 0 && p < cap, NC_ERR_POSITION, "position %d of sequence %d outside [0, %d)", p,
             b, cap);
    if (kv->paged)
      for (int i = 0; i <= p / kv->block_size; ++i) {
        const int blk = kv->block_table_host[(size_t)b * kv->max_blocks_per_seq + i];
        NC_CHECK(blk >= 0 && blk < kv->num_blocks, NC_ERR_POSITION,
                 "block table entry %d of sequence %d is %d", i, b, blk);
      }
  }
  NC_CHECK(B * n_kv_heads <= kStaticAttnTickets, NC_ERR_CAPACITY,
           "batch x kv heads = %d exceeds the %d static merge tickets", B * n_kv_heads,
           kStaticAttnTickets);
  const int splits = attn_splits(B, n_kv_heads, head_dim, kv->dtype == NC_KV_BF16, cap);
  const size_t need = attn_part_floats(B, n_q_heads, head_dim, splits);
  NC_CHECK(need <= kStaticAttnScratchFloats, NC_ERR_CAPACITY,
           "attention needs %zu scratch floats (%d splits); the static array holds %zu", need,
           splits, kStaticAttnScratchFloats);

  float* scratch = nullptr;
  unsigned int* tickets = nullptr;
  int* status = nullptr;
  cudaError_t e = static_scratch(static_cast<cudaStream_t>(stream), &scratch, &tickets, &status);
  if (e != cudaSuccess)
    return fail(NC_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                cudaGetErrorString(e));
  KVView v;
  v.k = kv->k;
  v.v = kv->v;
  v.block_table = kv->block_table;
  v.paged = kv->paged;
  v.bf16 = kv->dtype == NC_KV_BF16;
  v.batch_capacity = kv->batch_capacity;
  v.max_ctx = kv->max_ctx;
  v.block_size = kv->block_size;
  v.num_blocks = kv->num_blocks;
  v.max_blocks_per_seq = kv->max_blocks_per_seq;
  v.n_kv_heads = n_kv_heads;
  v.head_dim = head_dim;
  AttnArgs a{q, positions_dev, B, n_q_heads, n_kv_heads, head_dim, layer, splits, scratch, out, v,
             status, tickets};
  e = launch_attn(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(NC_ERR_CUDA, "nc_attn_decode_static: %s", cudaGetErrorString(e));
  return NC_OK;
}

extern "C" nc_status nc_attn_decode_static_status(void* stream, int* code) {
  NC_CHECK(code, NC_ERR_INVALID_ARGUMENT, "code is NULL");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  const int zero = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&word, g_attn_status, sizeof(int));
  if (e == cudaSuccess && word != 0) e = cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int));
  if (e != cudaSuccess)
    return fail(NC_ERR_CUDA, "reading the static attention status failed: %s",
                cudaGetErrorString(e));
  *code = word;
  return NC_OK;
}
