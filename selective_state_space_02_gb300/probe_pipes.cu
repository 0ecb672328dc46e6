// Pipe-rate probe for the ALU roofline of the scan: issue-limited throughput
// of FFMA, packed FFMA2/FMUL2 (f32x2), and the special-function unit (ex2,
// lg2, rcp, tanh) on the current GPU, per SM per nanosecond.  Each thread runs
// 8 independent chains; rates at 8, 16 and 32 warps per SM.
// Build and run:  nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o probe_pipes probe_pipes.cu && ./probe_pipes
#include <cstdio>
#include <cuda_runtime.h>
#define CK(x) do{cudaError_t e=(x); if(e!=cudaSuccess){printf("ERR %s @%d\n",cudaGetErrorString(e),__LINE__); return 1;}}while(0)

__device__ __forceinline__ unsigned long long pk(float a, float b){unsigned long long r; asm("mov.b64 %0, {%1,%2};":"=l"(r):"f"(a),"f"(b)); return r;}
__device__ __forceinline__ void upk(unsigned long long r, float&a, float&b){asm("mov.b64 {%0,%1}, %2;":"=f"(a),"=f"(b):"l"(r));}

template<int MODE>
__global__ void k(float* out, int iters, float s) {
  float v[8]; unsigned long long p[8];
  for (int i=0;i<8;i++){ v[i]= 0.001f*(threadIdx.x+i); p[i]=pk(v[i], v[i]+0.5f);} 
  unsigned long long ps = pk(s, s);
  for (int it=0; it<iters; ++it) {
#pragma unroll
    for (int i=0;i<8;i++){
      if (MODE==0) { v[i] = fmaf(v[i], s, 0.25f); }
      else if (MODE==1) { asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(p[i]) : "l"(ps), "l"(ps)); }
      else if (MODE==2) { asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(v[i])); v[i] = -v[i]; }
      else if (MODE==3) { float t; asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(v[i])); v[i] = fmaf(t, s, -0.5f); v[i]=fmaf(v[i],s,0.1f);} 
      else if (MODE==4) { float t; asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(v[i])); unsigned long long q=pk(t,t); asm volatile("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(p[i]) : "l"(q), "l"(ps)); v[i] = -t; }
      else if (MODE==5) { float t; asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(v[i]+2.0f)); v[i]=t; }
      else if (MODE==6) { float t; asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(v[i]+2.0f)); v[i]=t; }
      else if (MODE==7) { asm volatile("mul.rn.f32x2 %0, %0, %1;" : "+l"(p[i]) : "l"(ps)); }
      else if (MODE==8) { float t; asm volatile("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(v[i])); v[i]=t; }
    }
  }
  float acc=0; for(int i=0;i<8;i++){ float a,b; upk(p[i],a,b); acc+=v[i]+a+b; }
  if (acc == 1234.5f) out[threadIdx.x]=acc;
}

int main(){
  int dev=0; cudaDeviceProp pr; CK(cudaGetDeviceProperties(&pr,dev));
  int clk=0; cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev);
  printf("GPU %s SMs %d clockRate(kHz) %d smemPerBlockOptin %zu L2 %d regsPerSM %d\n", pr.name, pr.multiProcessorCount, clk, pr.sharedMemPerBlockOptin, pr.l2CacheSize, pr.regsPerMultiprocessor);
  float* out; CK(cudaMalloc(&out, 4096));
  const char* names[]={"FFMA","FFMA2(f32x2)","EX2","EX2+2FFMA","EX2+FFMA2","LG2","RCP","FMUL2","TANH"};
  cudaEvent_t a,b; cudaEventCreate(&a); cudaEventCreate(&b);
  int sms=pr.multiProcessorCount;
  for (int warps=8; warps<=32; warps*=2) {
  for (int m=0;m<9;m++){
    int threads=warps*32/ 1; int blocks=sms*1; int iters=4096;
    void (*f)(float*,int,float);
    switch(m){case 0:f=k<0>;break;case 1:f=k<1>;break;case 2:f=k<2>;break;case 3:f=k<3>;break;case 4:f=k<4>;break;case 5:f=k<5>;break;case 6:f=k<6>;break;case 7:f=k<7>;break;default:f=k<8>;}
    for(int w=0;w<2;w++) f<<<blocks,threads>>>(out,iters,0.999f);
    CK(cudaDeviceSynchronize());
    cudaEventRecord(a); f<<<blocks,threads>>>(out,iters,0.999f); cudaEventRecord(b); CK(cudaEventSynchronize(b));
    float ms; cudaEventElapsedTime(&ms,a,b);
    double ops = (double)blocks*threads*iters*8; // "op units" per thread-iteration-chain
    printf("warps/SM %2d %-14s %.3f ms  %.3f Tunit/s  per-SM-per-ns %.2f\n", warps, names[m], ms, ops/ms/1e9, ops/ms/1e6/sms);
  }}
  return 0;
}
