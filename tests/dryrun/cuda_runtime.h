// A stand-in for the CUDA runtime header, used only by the host-only dry-run
// build of the step executor (tests/dryrun): the executor's C++ compiles
// against these declarations with g++, and dryrun.cpp implements them by
// recording streams, events and the memory each launch touches, so that the
// tests can check the executor's ordering and bounds without a GPU.
// It declares only what the executor's translation unit uses.
#pragma once
#include <stddef.h>
#include <stdint.h>

#define __device__
#define __forceinline__ inline
#define __global__

typedef int cudaError_t;
enum : int { cudaSuccess = 0, cudaErrorInvalidValue = 1 };

struct CUstream_st;
typedef CUstream_st* cudaStream_t;
struct CUevent_st;
typedef CUevent_st* cudaEvent_t;
struct CUgraph_st;
typedef CUgraph_st* cudaGraph_t;
struct CUgraphExec_st;
typedef CUgraphExec_st* cudaGraphExec_t;

struct dim3 {
  unsigned x, y, z;
  dim3(unsigned a = 1, unsigned b = 1, unsigned c = 1) : x(a), y(b), z(c) {}
};

enum cudaStreamCaptureStatus {
  cudaStreamCaptureStatusNone = 0,
  cudaStreamCaptureStatusActive = 1,
  cudaStreamCaptureStatusInvalidated = 2
};
enum cudaStreamCaptureMode {
  cudaStreamCaptureModeGlobal = 0,
  cudaStreamCaptureModeThreadLocal = 1,
  cudaStreamCaptureModeRelaxed = 2
};
enum cudaMemcpyKind {
  cudaMemcpyHostToHost = 0,
  cudaMemcpyHostToDevice = 1,
  cudaMemcpyDeviceToHost = 2,
  cudaMemcpyDeviceToDevice = 3,
  cudaMemcpyDefault = 4
};
#define cudaStreamNonBlocking 0x01
#define cudaEventDisableTiming 0x02
#define cudaEventRecordExternal 0x01
#define cudaGraphInstantiateFlagUseNodePriority 8

enum cudaLaunchAttributeID {
  cudaLaunchAttributeProgrammaticStreamSerialization = 5,
  cudaLaunchAttributePriority = 8
};
union cudaLaunchAttributeValue {
  int priority;
  int programmaticStreamSerializationAllowed;
  char pad[64];
};
struct cudaLaunchAttribute {
  cudaLaunchAttributeID id;
  cudaLaunchAttributeValue val;
};
struct cudaLaunchConfig_t {
  dim3 gridDim;
  dim3 blockDim;
  size_t dynamicSmemBytes;
  cudaStream_t stream;
  cudaLaunchAttribute* attrs;
  unsigned numAttrs;
};

template <typename... A>
cudaError_t cudaLaunchKernelEx(const cudaLaunchConfig_t*, A...) {
  return cudaErrorInvalidValue;  // the dry run launches no kernel itself
}

const char* cudaGetErrorString(cudaError_t e);
cudaError_t cudaGetDevice(int* dev);
cudaError_t cudaDeviceGetStreamPriorityRange(int* least, int* greatest);
cudaError_t cudaStreamCreateWithFlags(cudaStream_t* s, unsigned flags);
cudaError_t cudaStreamCreateWithPriority(cudaStream_t* s, unsigned flags, int priority);
cudaError_t cudaStreamGetPriority(cudaStream_t s, int* priority);
cudaError_t cudaStreamDestroy(cudaStream_t s);
cudaError_t cudaStreamSynchronize(cudaStream_t s);
cudaError_t cudaStreamWaitEvent(cudaStream_t s, cudaEvent_t e, unsigned flags);
cudaError_t cudaStreamBeginCapture(cudaStream_t s, cudaStreamCaptureMode mode);
cudaError_t cudaStreamEndCapture(cudaStream_t s, cudaGraph_t* g);
cudaError_t cudaStreamIsCapturing(cudaStream_t s, cudaStreamCaptureStatus* status);
cudaError_t cudaEventCreate(cudaEvent_t* e);
cudaError_t cudaEventCreateWithFlags(cudaEvent_t* e, unsigned flags);
cudaError_t cudaEventDestroy(cudaEvent_t e);
cudaError_t cudaEventRecord(cudaEvent_t e, cudaStream_t s = nullptr);
cudaError_t cudaEventRecordWithFlags(cudaEvent_t e, cudaStream_t s, unsigned flags);
cudaError_t cudaEventSynchronize(cudaEvent_t e);
cudaError_t cudaEventElapsedTime(float* ms, cudaEvent_t a, cudaEvent_t b);
cudaError_t cudaGraphInstantiate(cudaGraphExec_t* exec, cudaGraph_t g, unsigned long long flags);
cudaError_t cudaGraphLaunch(cudaGraphExec_t exec, cudaStream_t s);
cudaError_t cudaGraphDestroy(cudaGraph_t g);
cudaError_t cudaGraphExecDestroy(cudaGraphExec_t exec);
cudaError_t cudaMemsetAsync(void* p, int value, size_t bytes, cudaStream_t s = nullptr);
cudaError_t cudaMemcpyAsync(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s = nullptr);
