// tc_loop_floor: the launch floor of the device-resident decode loop.
//
// "Constraint made cheaper than no constraint" separates the cost of adding a
// kernel from the cost of the work it does by launching a do-nothing kernel
// in the sampler's place.  This builds tc_decode's graph shape with such a
// kernel in the step's place: a reset kernel that arms the loop, then a
// conditional WHILE node whose body holds kLoopUnroll launches of the
// one-CTA-per-sequence step grid (1, batch) x 256 threads, chained with
// programmatic dependent launch; the body's last launch sets the loop
// condition from a device counter.  The time per launch is the least a
// decode step of that shape can cost in this loop.
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "kernels.h"
#include "tcd.h"
#include "tcd_internal.h"

namespace {

__global__ void floor_arm_kernel(int32_t* left, int32_t iterations, unsigned long long cond) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    *left = iterations;
    cudaGraphSetConditional((cudaGraphConditionalHandle)cond, iterations > 0 ? 1u : 0u);
  }
}

// Does nothing but wait for its predecessor and let its successor launch;
// the body's last launch counts the iteration and sets the loop condition.
__global__ void __launch_bounds__(tcd::kThreads) floor_step_kernel(int32_t* left, int32_t loop_ctrl,
                                                                   unsigned long long cond) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (loop_ctrl && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) {
    const int32_t l = *left - 1;
    *left = l;
    cudaGraphSetConditional((cudaGraphConditionalHandle)cond, l > 0 ? 1u : 0u);
  }
}

cudaError_t launch_floor_step(int32_t batch, int32_t* left, int32_t loop_ctrl, unsigned long long cond, bool pdl,
                              cudaStream_t s) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(1, batch);
  cfg.blockDim = dim3(tcd::kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, floor_step_kernel, left, loop_ctrl, cond);
}

struct FloorState {
  cudaStream_t cs = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaEvent_t a = nullptr, b = nullptr;
  int32_t* left = nullptr;
  ~FloorState() {
    if (exec) cudaGraphExecDestroy(exec);
    if (graph) cudaGraphDestroy(graph);
    if (a) cudaEventDestroy(a);
    if (b) cudaEventDestroy(b);
    if (left) cudaFree(left);
    if (cs) cudaStreamDestroy(cs);
  }
};

tc_status floor_fail(cudaError_t e, const char* what) {
  tcd::set_error_message(std::string("tc_loop_floor: ") + what + ": " + cudaGetErrorString(e));
  cudaGetLastError();
  return TC_ERR_CUDA;
}

}  // namespace

extern "C" tc_status tc_loop_floor(int32_t device, int32_t batch, int32_t iterations, void* stream, float* ms_out,
                                   int64_t* launches_out) {
  if (!ms_out || !launches_out || batch < 1 || batch > 65535 || iterations < 1) {
    tcd::set_error_message("tc_loop_floor: invalid arguments");
    return TC_ERR_INVALID_ARG;
  }
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return floor_fail(cudaGetLastError(), "cudaGetDevice");
  if (cudaSetDevice(device) != cudaSuccess) return floor_fail(cudaGetLastError(), "cudaSetDevice");
  tc_status rc = TC_OK;
  {
    FloorState f;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaGraphConditionalHandle cond = 0;
    cudaError_t e;
    auto fail = [&](cudaError_t err, const char* what) {
      cudaStreamCaptureStatus st;
      if (f.cs && cudaStreamIsCapturing(f.cs, &st) == cudaSuccess && st != cudaStreamCaptureStatusNone) {
        cudaGraph_t junk = nullptr;
        cudaStreamEndCapture(f.cs, &junk);
      }
      return floor_fail(err, what);
    };
    if ((e = cudaStreamCreateWithFlags(&f.cs, cudaStreamNonBlocking)) != cudaSuccess) rc = fail(e, "stream");
    if (rc == TC_OK && (e = cudaMalloc(&f.left, sizeof(int32_t))) != cudaSuccess) rc = fail(e, "counter");
    if (rc == TC_OK && (e = cudaGraphCreate(&f.graph, 0)) != cudaSuccess) rc = fail(e, "cudaGraphCreate");
    if (rc == TC_OK && (e = cudaGraphConditionalHandleCreate(&cond, f.graph, 0, 0)) != cudaSuccess)
      rc = fail(e, "cudaGraphConditionalHandleCreate");
    if (rc == TC_OK && (e = cudaStreamBeginCaptureToGraph(f.cs, f.graph, nullptr, nullptr, 0,
                                                          cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
      rc = fail(e, "capture");
    if (rc == TC_OK) {
      floor_arm_kernel<<<1, 32, 0, f.cs>>>(f.left, iterations, (unsigned long long)cond);
      if ((e = cudaGetLastError()) != cudaSuccess) rc = fail(e, "arm kernel");
    }
    cudaGraph_t body = nullptr;
    if (rc == TC_OK) {
      cudaStreamCaptureStatus cst;
      cudaGraph_t cap = nullptr;
      const cudaGraphNode_t* deps = nullptr;
      const cudaGraphEdgeData* edata = nullptr;
      size_t ndeps = 0;
      if ((e = cudaStreamGetCaptureInfo(f.cs, &cst, nullptr, &cap, &deps, &edata, &ndeps)) != cudaSuccess) {
        rc = fail(e, "cudaStreamGetCaptureInfo");
      } else {
        cudaGraphNodeParams np{};
        np.type = cudaGraphNodeTypeConditional;
        np.conditional.handle = cond;
        np.conditional.type = cudaGraphCondTypeWhile;
        np.conditional.size = 1;
        cudaGraphNode_t cnode = nullptr;
        if ((e = cudaGraphAddNode(&cnode, cap, deps, edata, ndeps, &np)) != cudaSuccess) {
          rc = fail(e, "conditional node");
        } else {
          body = np.conditional.phGraph_out[0];
          if ((e = cudaStreamUpdateCaptureDependencies(f.cs, &cnode, nullptr, 1,
                                                       cudaStreamSetCaptureDependencies)) != cudaSuccess)
            rc = fail(e, "capture dependencies");
        }
      }
      cudaGraph_t ended = nullptr;
      if (rc == TC_OK && (e = cudaStreamEndCapture(f.cs, &ended)) != cudaSuccess) rc = fail(e, "end capture");
    }
    if (rc == TC_OK && (e = cudaStreamBeginCaptureToGraph(f.cs, body, nullptr, nullptr, 0,
                                                          cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
      rc = fail(e, "body capture");
    for (int u = 0; rc == TC_OK && u < tcd::kLoopUnroll; ++u) {
      if ((e = launch_floor_step(batch, f.left, u == tcd::kLoopUnroll - 1, (unsigned long long)cond, u > 0,
                                 f.cs)) != cudaSuccess)
        rc = fail(e, "step capture");
    }
    if (rc == TC_OK) {
      cudaGraph_t ended = nullptr;
      if ((e = cudaStreamEndCapture(f.cs, &ended)) != cudaSuccess) rc = fail(e, "end body capture");
    }
    if (rc == TC_OK && (e = cudaGraphInstantiate(&f.exec, f.graph, 0)) != cudaSuccess) rc = fail(e, "instantiate");
    if (rc == TC_OK && (e = cudaEventCreate(&f.a)) != cudaSuccess) rc = fail(e, "event");
    if (rc == TC_OK && (e = cudaEventCreate(&f.b)) != cudaSuccess) rc = fail(e, "event");
    // one untimed launch, then the timed one
    if (rc == TC_OK && (e = cudaGraphLaunch(f.exec, s)) != cudaSuccess) rc = fail(e, "warm-up launch");
    if (rc == TC_OK && (e = cudaEventRecord(f.a, s)) != cudaSuccess) rc = fail(e, "event record");
    if (rc == TC_OK && (e = cudaGraphLaunch(f.exec, s)) != cudaSuccess) rc = fail(e, "launch");
    if (rc == TC_OK && (e = cudaEventRecord(f.b, s)) != cudaSuccess) rc = fail(e, "event record");
    if (rc == TC_OK && (e = cudaEventSynchronize(f.b)) != cudaSuccess) rc = fail(e, "synchronize");
    float ms = 0.f;
    if (rc == TC_OK && (e = cudaEventElapsedTime(&ms, f.a, f.b)) != cudaSuccess) rc = fail(e, "elapsed time");
    if (rc == TC_OK) {
      *ms_out = ms;
      *launches_out = (int64_t)iterations * tcd::kLoopUnroll;
    }
    cudaStreamSynchronize(s);
  }
  cudaSetDevice(prev);
  return rc;
}
