// decode.cu -- host side of the decode attention kernel (decode_kernel.cuh):
// the geometry dispatch, the workspace size and the Qwen3 decoder's
// instantiation (16 query / 8 KV heads of dimension 128, head counts fixed at
// compile time). The instantiations for run-time head counts are built in
// decode_d64.cu and decode_d128.cu, so that the three translation units
// compile in parallel.
#include "decode_kernel.cuh"

namespace pkv {

int decode_max_batch() { return kMaxDecodeBatch; }

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}
}  // namespace

int encode_page_maps(const void* k_pages, const void* v_pages, int head_dim, int num_pages, int hkv, CUtensorMap* kmap,
                     CUtensorMap* vmap) {
  const long long tiles = static_cast<long long>(num_pages) * hkv;
  if (tiles > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // tile coordinates are 32-bit
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return PKV_ERR_CUDA;
  const cuuint32_t halves = static_cast<cuuint32_t>(head_dim / 64);
  // (dim within the half, row, half, tile): a tile's halves are 128 bytes apart inside each 2 * head_dim-byte row
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(kPageSize), halves, static_cast<cuuint64_t>(tiles)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(head_dim) * 2, 128,
                                 static_cast<cuuint64_t>(head_dim) * 2 * kPageSize};
  const cuuint32_t box[4] = {64, kPageSize, halves, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const void* pools[2] = {k_pages, v_pages};
  CUtensorMap* maps[2] = {kmap, vmap};
  for (int i = 0; i < 2; ++i)
    if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pools[i]), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PKV_ERR_CUDA;
  return PKV_OK;
}

// The kernel's group for g query heads per KV head: the next of 1, 2, 4, 8.
static int group_pad(int g) { return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8; }

static bool fixed_geometry(int hq, int hkv, int head_dim) {
  return hq == kQHeads && hkv == kKVHeads && head_dim == kHeadDim;
}

bool decode_supported(int num_q_heads, int num_kv_heads, int head_dim, int page_size) {
  if (num_kv_heads < 1 || num_kv_heads > 65535 || page_size != kPageSize) return false;
  if (num_q_heads % num_kv_heads != 0) return false;
  const int g = num_q_heads / num_kv_heads;
  return g >= 1 && g <= 8 && (head_dim == 64 || head_dim == 128);
}

size_t decode_workspace_bytes(int num_q_heads, int num_kv_heads, int head_dim, int32_t batch, int num_sms) {
  const size_t G = static_cast<size_t>(group_pad(num_q_heads / num_kv_heads));
  const size_t grid = static_cast<size_t>(decode_grid(num_sms));
  size_t off = PKV_STATUS_BYTES + decode_counter_bytes(batch, num_kv_heads);
  off += 2 * grid * G * (head_dim + 4) * 4;      // counted records
  off += 2 * grid * (G * head_dim + 4 * G) * 4;  // polled records
  return off;
}

int launch_decode(const void* q, const void* k_new, const void* v_new, const void* k_pages, const void* v_pages,
                  const int32_t* block_table, const int32_t* seq_lens, const float* rope, int32_t rope_max_pos,
                  void* out, float scale, int num_q_heads, int num_kv_heads, int head_dim, int32_t batch,
                  int32_t max_pages, int32_t num_pages, void* workspace, int num_sms, cudaStream_t stream,
                  uint32_t flags) {
  if (!decode_supported(num_q_heads, num_kv_heads, head_dim, kPageSize)) return PKV_ERR_UNSUPPORTED;
  DecodeLaunch c;
  c.q = q;
  c.k_new = k_new;
  c.v_new = v_new;
  c.k_pages = k_pages;
  c.v_pages = v_pages;
  c.block_table = block_table;
  c.seq_lens = seq_lens;
  c.rope = rope;
  c.rope_max_pos = rope_max_pos;
  c.out = out;
  c.scale = scale;
  c.hq = num_q_heads;
  c.hkv = num_kv_heads;
  c.head_dim = head_dim;
  c.batch = batch;
  c.max_pages = max_pages;
  c.num_pages = num_pages;
  c.workspace = workspace;
  c.num_sms = num_sms;
  c.stream = stream;
  c.flags = flags;
  if (fixed_geometry(num_q_heads, num_kv_heads, head_dim)) return launch_decode_geo<DecGeo<128, 2, true>>(c);
  const int G = group_pad(num_q_heads / num_kv_heads);
  return head_dim == 64 ? launch_decode_d64(c, G) : launch_decode_d128(c, G);
}

}  // namespace pkv
