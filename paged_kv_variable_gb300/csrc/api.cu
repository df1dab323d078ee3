// C-ABI entry points: argument validation, TMA descriptors, launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kernels.h"

namespace pkv {

namespace {
thread_local char g_err[512] = "";
thread_local cudaEvent_t g_ev_start = nullptr;
thread_local cudaEvent_t g_ev_stop = nullptr;

// Under stream capture the record becomes an event-record node of the graph,
// so that every replay re-records the caller's event around the kernel.
cudaError_t record_profile_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, s);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

pkv_status fail(pkv_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

pkv_status validate_problem(const pkv_problem* p);  // plan.cpp

namespace {

pkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// 4-D map over a cache (D, Hkv, rows-per-page-or-seq, pages-or-batch); a box
// is cache_box_rows() rows of one 128-byte column chunk with the 128-byte
// swizzle (an fp8 cache at D = 64: its 64-byte rows with the 64-byte swizzle),
// zero fill outside the tensor.
pkv_status make_cache_map(CUtensorMap* map, const pkv_problem& pr, const pkv_fwd_args& a, void* base) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const bool fp8 = pr.cache_dtype == PKV_FP8_E4M3;
  const int es = fp8 ? 1 : 2;
  const cuuint64_t rows = pr.page_size > 0 ? (cuuint64_t)pr.page_size : (cuuint64_t)pr.cache_capacity;
  cuuint64_t dims[4] = {(cuuint64_t)pr.head_dim, (cuuint64_t)pr.num_heads_kv, rows, (cuuint64_t)pr.num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)a.kc_stride_head * es, (cuuint64_t)a.kc_stride_tok * es,
                           (cuuint64_t)a.kc_stride_page * es};
  cuuint32_t box[4] = {(cuuint32_t)(128 / es), 1,
                       (cuuint32_t)cache_box_rows(pr.page_size, pr.cache_capacity, kv_tile_keys(pr.head_dim)), 1};
  const bool narrow = pr.head_dim * es < 128;
  if (narrow) box[0] = (cuuint32_t)pr.head_dim;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PKV_OK;
}

// 3-D map over q (D, Hq, total_q): a box of nh heads x 128/nh tokens (nh = G,
// at most 128) is the Q tile of one tensor-core item (row = token * nh + g).
pkv_status make_q_map(CUtensorMap* map, const pkv_problem& pr, const pkv_fwd_args& a, int total_q) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int nh = tc_group_heads(pr.num_heads_q / pr.num_heads_kv);
  cuuint64_t dims[3] = {(cuuint64_t)pr.head_dim, (cuuint64_t)pr.num_heads_q, (cuuint64_t)(total_q > 0 ? total_q : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)a.q_stride_head * 2, (cuuint64_t)a.q_stride_tok * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)nh, (cuuint32_t)(kPrefillRowsTc / nh)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed (%d)", (int)r);
  return PKV_OK;
}

pkv_status validate_cache_args(const pkv_problem& pr, const pkv_fwd_args* a) {
  if (!a) return fail(PKV_ERR_INVALID_ARG, "args is NULL");
  if (!a->k_cache || !a->v_cache) return fail(PKV_ERR_INVALID_ARG, "k_cache / v_cache is NULL");
  if (!aligned16(a->k_cache) || !aligned16(a->v_cache))
    return fail(PKV_ERR_INVALID_ARG, "cache base pointers must be 16-byte aligned");
  if (!a->cache_seqlens) return fail(PKV_ERR_INVALID_ARG, "cache_seqlens is NULL");
  const int es = pr.cache_dtype == PKV_FP8_E4M3 ? 1 : 2;
  if (a->kc_stride_head <= 0 || a->kc_stride_tok <= 0 || a->kc_stride_page <= 0)
    return fail(PKV_ERR_INVALID_ARG, "cache strides must be positive");
  if ((a->kc_stride_head * es) % 16 || (a->kc_stride_tok * es) % 16 || (a->kc_stride_page * es) % 16)
    return fail(PKV_ERR_INVALID_ARG, "cache strides must be multiples of 16 bytes");
  if (a->kc_stride_head < pr.head_dim) return fail(PKV_ERR_INVALID_ARG, "kc_stride_head < head_dim");
  if (pr.page_size > 0) {
    if (!a->block_table) return fail(PKV_ERR_INVALID_ARG, "paged cache needs block_table");
    if (!a->page_indptr && a->block_table_stride < pr.cache_capacity / pr.page_size)
      return fail(PKV_ERR_INVALID_ARG, "block_table_stride %d < cache_capacity / page_size", a->block_table_stride);
  }
  if (pr.cache_dtype == PKV_FP8_E4M3 && (!a->k_scale || !a->v_scale))
    return fail(PKV_ERR_INVALID_ARG, "fp8 cache needs k_scale and v_scale");
  return PKV_OK;
}

pkv_status validate_new_args(const pkv_problem& pr, const pkv_fwd_args* a) {
  if (!a->k_new || !a->v_new || !a->cu_seqlens_knew)
    return fail(PKV_ERR_INVALID_ARG, "k_new, v_new and cu_seqlens_knew must all be given");
  if (!aligned16(a->k_new) || !aligned16(a->v_new))
    return fail(PKV_ERR_INVALID_ARG, "k_new / v_new must be 16-byte aligned");
  if (a->knew_stride_head < pr.head_dim || a->knew_stride_tok <= 0 || (a->knew_stride_head * 2) % 16 ||
      (a->knew_stride_tok * 2) % 16)
    return fail(PKV_ERR_INVALID_ARG, "k_new strides must be >= head_dim and multiples of 16 bytes");
  return PKV_OK;
}

AppendParams append_params(const pkv_problem& pr, const pkv_fwd_args* a, int32_t total_new, int* status) {
  AppendParams ap{};
  ap.k_new = static_cast<const __nv_bfloat16*>(a->k_new);
  ap.v_new = static_cast<const __nv_bfloat16*>(a->v_new);
  ap.n_stride_tok = a->knew_stride_tok;
  ap.n_stride_head = a->knew_stride_head;
  ap.cu_knew = a->cu_seqlens_knew;
  ap.cache_seqlens = a->cache_seqlens;
  ap.k_cache = a->k_cache;
  ap.v_cache = a->v_cache;
  ap.c_stride_page = a->kc_stride_page;
  ap.c_stride_tok = a->kc_stride_tok;
  ap.c_stride_head = a->kc_stride_head;
  ap.block_table = a->block_table;
  ap.bt_stride = a->block_table_stride;
  ap.page_indptr = a->page_indptr;
  ap.page_size = pr.page_size;
  ap.num_pages = pr.num_pages;
  ap.capacity = pr.cache_capacity;
  ap.batch = pr.batch;
  ap.hkv = pr.num_heads_kv;
  ap.total_new = total_new;
  ap.k_scale = a->k_scale;
  ap.v_scale = a->v_scale;
  ap.status = status;
  return ap;
}

bool same_problem(const pkv_problem& x, const pkv_problem& y) {
  return x.batch == y.batch && x.num_heads_q == y.num_heads_q && x.num_heads_kv == y.num_heads_kv &&
         x.head_dim == y.head_dim && x.page_size == y.page_size && x.cache_capacity == y.cache_capacity &&
         x.num_pages == y.num_pages && x.cache_dtype == y.cache_dtype && x.causal == y.causal &&
         x.softmax_scale == y.softmax_scale;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" const char* pkv_last_error(void) { return g_err; }

extern "C" const char* pkv_version(void) { return "pkv 0.1.0 (sm_103a)"; }

extern "C" pkv_status pkv_plan_upload(pkv_plan_t plan, void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan || !workspace) return fail(PKV_ERR_INVALID_ARG, "NULL plan or workspace");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan->layout.total)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu required", workspace_bytes, plan->layout.total);
  cudaError_t e = cudaMemcpyAsync(workspace, plan->image, plan->image_bytes, cudaMemcpyHostToDevice,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "plan upload");
  return PKV_OK;
}

extern "C" pkv_status pkv_kv_append(const pkv_problem* problem, const pkv_fwd_args* args, int32_t total_new,
                                    int32_t* device_status, void* stream) {
  pkv_status st = validate_problem(problem);
  if (st != PKV_OK) return st;
  st = validate_cache_args(*problem, args);
  if (st != PKV_OK) return st;
  if (total_new < 0) return fail(PKV_ERR_INVALID_ARG, "total_new < 0");
  if (total_new == 0) return PKV_OK;
  st = validate_new_args(*problem, args);
  if (st != PKV_OK) return st;
  AppendParams ap = append_params(*problem, args, total_new, reinterpret_cast<int*>(device_status));
  cudaError_t e = launch_kv_append(ap, problem->head_dim, problem->cache_dtype == PKV_FP8_E4M3,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return PKV_OK;
}

namespace pkv {

// Every host-side check of an attention call that does not involve the
// workspace: the problem, the plan it must match, the cache, q / out and the
// new-token arguments.  Nothing is launched or copied before these pass.
pkv_status validate_call(const pkv_problem* problem, const pkv_fwd_args* args, pkv_plan_t plan) {
  pkv_status st = validate_problem(problem);
  if (st != PKV_OK) return st;
  if (!plan) return fail(PKV_ERR_INVALID_ARG, "plan is NULL");
  if (!same_problem(*problem, plan->problem)) return fail(PKV_ERR_INVALID_ARG, "problem differs from the plan's");
  st = validate_cache_args(*problem, args);
  if (st != PKV_OK) return st;
  const pkv_problem& pr = *problem;
  if (plan->total_q > 0) {
    if (!args->q || !args->out || !args->cu_seqlens_q) return fail(PKV_ERR_INVALID_ARG, "q, out or cu_seqlens_q NULL");
    if (args->q_stride_head < pr.head_dim || args->o_stride_head < pr.head_dim || args->q_stride_tok <= 0 ||
        args->o_stride_tok <= 0)
      return fail(PKV_ERR_INVALID_ARG, "q / out strides");
    if (!aligned16(args->q) || !aligned16(args->out) || (args->q_stride_head % 8) || (args->q_stride_tok % 8) ||
        (args->o_stride_head % 8) || (args->o_stride_tok % 8))
      return fail(PKV_ERR_INVALID_ARG, "q / out must be 16-byte aligned with strides multiple of 8 elements");
    if (args->max_seqlen_q < 0) return fail(PKV_ERR_INVALID_ARG, "max_seqlen_q < 0");
    if (args->q_rows != 0 && args->q_rows < plan->total_q)
      return fail(PKV_ERR_INVALID_ARG, "q_rows %d < the plan's %d query rows", args->q_rows, plan->total_q);
  }
  if (args->q_rows < 0) return fail(PKV_ERR_INVALID_ARG, "q_rows < 0");
  const bool has_new = args->k_new != nullptr || args->v_new != nullptr;
  if (plan->total_new > 0 && !has_new)
    return fail(PKV_ERR_INVALID_ARG, "the plan appends %d tokens but k_new / v_new are NULL", plan->total_new);
  if (plan->total_new == 0 && has_new)
    return fail(PKV_ERR_INVALID_ARG, "k_new given but the plan was made with no new tokens");
  if (plan->total_new > 0) {
    st = validate_new_args(pr, args);
    if (st != PKV_OK) return st;
  }
  if (args->q_scale && pr.cache_dtype != PKV_FP8_E4M3)
    return fail(PKV_ERR_UNSUPPORTED, "q_scale (fp8 Q.K^T) needs an fp8 cache");
  return PKV_OK;
}

}  // namespace pkv

extern "C" pkv_status pkv_attn_varlen_kvcache_fwd(const pkv_problem* problem, const pkv_fwd_args* args,
                                                  pkv_plan_t plan, void* workspace, size_t workspace_bytes,
                                                  void* stream) {
  pkv_status st = validate_call(problem, args, plan);
  if (st != PKV_OK) return st;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(PKV_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
  if (workspace_bytes < plan->layout.total)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu required", workspace_bytes, plan->layout.total);
  const pkv_problem& pr = *problem;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  int* status = reinterpret_cast<int*>(ws + plan->layout.status);

  if (plan->total_new > 0) {
    AppendParams ap = append_params(pr, args, plan->total_new, status);
    cudaError_t e = launch_kv_append(ap, pr.head_dim, pr.cache_dtype == PKV_FP8_E4M3, s);
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  }
  if (plan->num_items == 0) return PKV_OK;

  CUtensorMap tk, tv, tq;
  st = make_cache_map(&tk, pr, *args, args->k_cache);
  if (st != PKV_OK) return st;
  st = make_cache_map(&tv, pr, *args, args->v_cache);
  if (st != PKV_OK) return st;
  memset(&tq, 0, sizeof(tq));
  if (plan->num_prefill_items > 0) {
    st = make_q_map(&tq, pr, *args, args->q_rows ? args->q_rows : plan->total_q);
    if (st != PKV_OK) return st;
  }

  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(args->q);
  p.q_stride_tok = args->q_stride_tok;
  p.q_stride_head = args->q_stride_head;
  p.out = static_cast<__nv_bfloat16*>(args->out);
  p.o_stride_tok = args->o_stride_tok;
  p.o_stride_head = args->o_stride_head;
  p.out_v8 = (reinterpret_cast<uintptr_t>(args->out) % 32 == 0) && (args->o_stride_tok % 16 == 0) &&
             (args->o_stride_head % 16 == 0);
  p.lse = args->lse;
  p.total_q = args->q_rows ? args->q_rows : plan->total_q;
  // rows placed by the caller (q_rows given): offsets read on the device
  p.q_offsets = args->q_rows ? args->cu_seqlens_q : nullptr;
  p.block_table = args->block_table;
  p.bt_stride = args->block_table_stride;
  p.page_indptr = args->page_indptr;
  p.page_size = pr.page_size;
  p.box_rows = cache_box_rows(pr.page_size, pr.cache_capacity, kv_tile_keys(pr.head_dim));
  p.num_pages = pr.num_pages;
  p.G = pr.num_heads_q / pr.num_heads_kv;
  p.causal = pr.causal;
  p.scale_log2 = pr.softmax_scale * 1.4426950408889634f;
  p.k_scale = args->k_scale;
  p.q_scale = args->q_scale;
  p.v_scale = args->v_scale;
  p.items = reinterpret_cast<const WorkItem*>(ws + plan->layout.items);
  p.cta_begin = reinterpret_cast<const int32_t*>(ws + plan->layout.cta_begin);
  p.partial_o = reinterpret_cast<float*>(ws + plan->layout.partial_o);
  p.partial_lse = reinterpret_cast<float*>(ws + plan->layout.partial_lse);
  p.status = status;
  p.cache_seqlens = args->cache_seqlens;
  p.plan_lc = reinterpret_cast<const int32_t*>(ws + plan->layout.plan_lc);
  p.batch = pr.batch;
  p.dynamic = plan->dynamic;
  p.row_gather = pr.page_size > 0 && pr.page_size < kBoxRows;
  p.kc = args->k_cache;
  p.vc = args->v_cache;
  p.c_stride_page = args->kc_stride_page;
  p.c_stride_tok = args->kc_stride_tok;
  p.c_stride_head = args->kc_stride_head;
  cudaError_t e;
  if (g_ev_start && (e = record_profile_event(g_ev_start, s)) != cudaSuccess) return cuda_fail(e, "profile event");
  // Decode-only plans overlap the attention kernel's start with the (small)
  // append kernel and the combine kernel's start with the attention's end.
  // Plans with prefill tiles keep the kernels strictly in order: there the
  // overlap measured slower (large appends, long attention kernels).  Never
  // across a profiling event, which must see the kernels in order.
  const bool overlap = plan->num_prefill_items == 0;
  e = launch_attention(p, tk, tv, tq, plan->num_ctas, pr.head_dim, pr.cache_dtype == PKV_FP8_E4M3,
                       plan->num_prefill_items > 0, plan->num_decode_items > 0,
                       overlap && plan->total_new > 0 && !g_ev_start, s);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  if (g_ev_stop && (e = record_profile_event(g_ev_stop, s)) != cudaSuccess) return cuda_fail(e, "profile event");

  if (plan->num_combine > 0) {
    CombineParams cp{};
    cp.items = reinterpret_cast<const CombineItem*>(ws + plan->layout.combine);
    cp.q_offsets = p.q_offsets;
    cp.partial_o = p.partial_o;
    cp.partial_lse = p.partial_lse;
    cp.out = p.out;
    cp.o_stride_tok = p.o_stride_tok;
    cp.o_stride_head = p.o_stride_head;
    cp.lse = p.lse;
    cp.total_q = p.total_q;
    cp.G = p.G;
    e = launch_combine(cp, plan->num_combine, pr.head_dim, overlap && !g_ev_stop, s);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  }
  return PKV_OK;
}

extern "C" pkv_status pkv_set_profile_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr))
    return fail(PKV_ERR_INVALID_ARG, "give both events or neither");
  g_ev_start = static_cast<cudaEvent_t>(start_event);
  g_ev_stop = static_cast<cudaEvent_t>(stop_event);
  return PKV_OK;
}

extern "C" pkv_status pkv_get_status(void* workspace, void* stream, int32_t* device_status) {
  if (!workspace || !device_status) return fail(PKV_ERR_INVALID_ARG, "NULL workspace or output");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h[4] = {0, 0, 0, 0};
  cudaError_t e = cudaMemcpyAsync(h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *device_status = h[0];
  if (h[0] != 0) {
    fail((pkv_status)h[0], "device status %d (info %d, %d)", h[0], h[1], h[2]);
    e = cudaMemsetAsync(workspace, 0, sizeof(h), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
  }
  return PKV_OK;
}
