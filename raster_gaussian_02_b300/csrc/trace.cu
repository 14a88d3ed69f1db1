// Kernel trace (include/gs2d.h, gs2d_trace_*): per-host-thread state behind
// the launch helper's event records, and the C entry points that turn it on
// and off and name the traced kernels.  Tracing changes no kernel and no
// result; it only adds two event records around each launch.
#include <cxxabi.h>

#include <cstdlib>
#include <cstring>

#include "gs2d_internal.cuh"

namespace gs2d {

namespace {

struct TraceThread {
  Trace t;
  const void* kernels[kTraceMaxKernels];
  char name[512];  // the last name handed out by gs2d_trace_kernel_name
};

TraceThread& tls() {
  static thread_local TraceThread s{};
  return s;
}

}  // namespace

Trace& trace_state() { return tls().t; }

void trace_set_kernel(int i, const void* kernel) {
  if (i >= 0 && i < kTraceMaxKernels) tls().kernels[i] = kernel;
}

cudaError_t trace_record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  const cudaError_t q = cudaStreamIsCapturing(s, &st);
  if (q != cudaSuccess) return q;
  return st == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal)
                                             : cudaEventRecord(e, s);
}

}  // namespace gs2d

extern "C" {

gs2d_status gs2d_trace_begin(const gs2d_event_t* events, int32_t max_kernels) {
  if (!events || max_kernels < 1 || max_kernels > gs2d::kTraceMaxKernels) return GS2D_ERR_INVALID_ARG;
  for (int32_t i = 0; i < 2 * max_kernels; ++i)
    if (!events[i]) return GS2D_ERR_INVALID_ARG;
  gs2d::Trace& t = gs2d::trace_state();
  t.events = reinterpret_cast<const cudaEvent_t*>(events);
  t.capacity = max_kernels;
  t.launched = 0;
  t.active = true;
  return GS2D_OK;
}

int32_t gs2d_trace_end(void) {
  gs2d::Trace& t = gs2d::trace_state();
  const int32_t n = t.active ? t.launched : 0;
  t.active = false;
  t.events = nullptr;
  return n;
}

const char* gs2d_trace_kernel_name(int32_t i) {
  gs2d::Trace& t = gs2d::trace_state();
  if (t.active || i < 0 || i >= t.capacity || i >= t.launched) return nullptr;
  const char* mangled = nullptr;
  if (cudaFuncGetName(&mangled, gs2d::tls().kernels[i]) != cudaSuccess || !mangled) return nullptr;
  int status = 0;
  char* dem = abi::__cxa_demangle(mangled, nullptr, nullptr, &status);
  const char* src = (status == 0 && dem) ? dem : mangled;
  // Demangled: "void ns::(anonymous namespace)::k_name<args>(params)".  Keep
  // "k_name<args>": drop the parameter list (the last top-level parenthesised
  // group) and everything up to the last "::" outside template arguments.
  size_t len = strlen(src), cut = len;
  if (dem) {
    int depth = 0;
    for (size_t k = len; k-- > 0;) {
      if (src[k] == ')') ++depth;
      if (src[k] == '(' && --depth == 0) {
        cut = k;
        break;
      }
    }
  }
  size_t from = 0;
  int angle = 0;
  for (size_t k = 0; k + 1 < cut; ++k) {
    if (src[k] == '<') ++angle;
    if (src[k] == '>') --angle;
    if (angle == 0 && src[k] == ':' && src[k + 1] == ':') from = k + 2;
  }
  char* out = gs2d::tls().name;
  const size_t cap = sizeof(gs2d::tls().name) - 1;
  const size_t m = cut - from < cap ? cut - from : cap;
  memcpy(out, src + from, m);
  out[m] = '\0';
  free(dem);
  return out;
}

}  // extern "C"
