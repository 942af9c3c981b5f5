// dispatch.cuh -- kernel selection by plan width and launch on the caller's stream.
#pragma once

#include "internal.h"

namespace rlca {

template <class Est>
struct WidthCaps {
  static constexpr int em = kEmMaxWidth;
  static constexpr int tm = kTmMaxWidth;
  static constexpr bool tm_fast = true;
};
template <bool H, class ST>
struct WidthCaps<RetraceEst<H, ST>> {
  static constexpr int em = kRetraceEmMaxWidth;
  static constexpr int tm = kRetraceTmMaxWidth;
  static constexpr bool tm_fast = false;  // stages its per-action blocks per tile
};

// smem = the driver's exchange arrays (sized here from the same shape
// constants and map type the kernel uses) + the estimator's staging bytes
template <class Est>
static cudaError_t launch_one(void (*kernel)(Est, Geom), const Plan& p, size_t smem, const Est& est,
                              const Geom& g, cudaStream_t s) {
  if (smem > kMaxSmemPerCta) return cudaErrorInvalidConfiguration;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.row_blocks * p.nseg));
  cfg.blockDim = dim3((unsigned)p.block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, est, g);
}

template <class Est, int W>
static cudaError_t launch_em_w(const Plan& p, const Est& est, const Geom& g, cudaStream_t s) {
  if constexpr (W <= WidthCaps<Est>::em) {
    using S = EmShape<W>;
    const size_t drv = S::NWR > 1 ? (size_t)2 * S::ROWS * S::NWR * sizeof(Aff<typename Est::V>) : 0;
    return launch_one<Est>(em_scan_kernel<Est, W>, p, drv + p.smem, est, g, s);
  } else {
    return cudaErrorInvalidConfiguration;
  }
}

template <class Est, int C>
static cudaError_t launch_tm_c(const Plan& p, const Est& est, const Geom& g, cudaStream_t s) {
  if constexpr (C <= WidthCaps<Est>::tm) {
    const size_t drv = (size_t)2 * C * 32 * sizeof(Aff<typename Est::V>);
    return launch_one<Est>(tm_scan_kernel<Est, C>, p, drv + p.smem, est, g, s);
  } else {
    return cudaErrorInvalidConfiguration;
  }
}

template <class Est, int W, int LS>
static cudaError_t launch_fast_wl(const Plan& p, const Est& est, const Geom& g, cudaStream_t s) {
  if constexpr (W <= WidthCaps<Est>::em) {
    using S = EmShape<W, LS>;
    const size_t drv = S::NWR > 1 ? (size_t)2 * S::ROWS * S::NWR * sizeof(Aff<typename Est::V>) : 0;
    return launch_one<Est>(em_fast_kernel<Est, W, LS>, p, drv + p.smem, est, g, s);
  } else {
    return cudaErrorInvalidConfiguration;
  }
}

template <class Est, int W>
static cudaError_t launch_fast_w(const Plan& p, const Est& est, const Geom& g, cudaStream_t s) {
  if (p.steps == 8) {
    if constexpr (W >= 32 || (sizeof(typename Est::Store) == 2 && W >= 8)) return launch_fast_wl<Est, W, 8>(p, est, g, s);
    return cudaErrorInvalidConfiguration;
  }
  return launch_fast_wl<Est, W, kEmSteps>(p, est, g, s);
}

template <class Est, int EW, int CT>
static cudaError_t launch_tf(const Plan& p, const Est& est, const Geom& g, cudaStream_t s) {
  if constexpr (WidthCaps<Est>::tm_fast) {
    return launch_one<Est>(tm_fast_kernel<Est, EW, CT>, p, tf_smem_bytes<typename Est::V, EW, CT>(), est, g, s);
  } else {
    return cudaErrorInvalidConfiguration;
  }
}

template <class Est, int EW, int CT>
static cudaError_t launch_ts(const Plan& p, const Est& est, const Geom& g, cudaStream_t s) {
  if constexpr (WidthCaps<Est>::tm_fast && Est::kStageable) {
    return launch_one<Est>(tm_staged_kernel<Est, EW, CT>, p, ts_smem_bytes<Est, EW, CT>(), est, g, s);
  } else {
    return cudaErrorInvalidConfiguration;
  }
}

template <class Est>
static cudaError_t launch_ts_any(const Plan& p, const Est& est, const Geom& g, cudaStream_t s) {
  if (p.env_width == 32) {
    switch (p.width) {
      case 1: return launch_ts<Est, 32, 1>(p, est, g, s);
      case 2: return launch_ts<Est, 32, 2>(p, est, g, s);
      case 4: return launch_ts<Est, 32, 4>(p, est, g, s);
      case 8: return launch_ts<Est, 32, 8>(p, est, g, s);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  if constexpr (sizeof(typename Est::Store) == 4) {
    if (p.env_width == 16) {
      switch (p.width) {
        case 4: return launch_ts<Est, 16, 4>(p, est, g, s);
        case 8: return launch_ts<Est, 16, 8>(p, est, g, s);
        case 16: return launch_ts<Est, 16, 16>(p, est, g, s);
        case 32: return launch_ts<Est, 16, 32>(p, est, g, s);
        default: return cudaErrorInvalidConfiguration;
      }
    }
  }
  return cudaErrorInvalidConfiguration;
}

template <class Est, int EW, int CT>
static cudaError_t launch_tb(const Plan& p, const Est& est, const Geom& g, cudaStream_t s, const TmaSet& maps) {
  if constexpr (WidthCaps<Est>::tm_fast && Est::kStageable) {
    void (*kernel)(Est, Geom, const TmaSet) = tm_bulk_kernel<Est, EW, CT>;
    const size_t smem = tb_smem_bytes<Est, EW, CT>();
    if (smem > kMaxSmemPerCta) return cudaErrorInvalidConfiguration;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.row_blocks * p.nseg));
    cfg.blockDim = dim3((unsigned)p.block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, est, g, maps);
  } else {
    return cudaErrorInvalidConfiguration;
  }
}

template <class Est>
static cudaError_t launch_tb_any(const Plan& p, const Est& est, const Geom& g, cudaStream_t s, const TmaSet& maps) {
  if constexpr (sizeof(typename Est::Store) == 4) {
    if (p.env_width == 8) {
      switch (p.width) {
        case 4: return launch_tb<Est, 8, 4>(p, est, g, s, maps);
        case 8: return launch_tb<Est, 8, 8>(p, est, g, s, maps);
        case 16: return launch_tb<Est, 8, 16>(p, est, g, s, maps);
        case 32: return launch_tb<Est, 8, 32>(p, est, g, s, maps);
        default: return cudaErrorInvalidConfiguration;
      }
    }
  }
  if (p.env_width == 16) {
    switch (p.width) {
      case 2: return launch_tb<Est, 16, 2>(p, est, g, s, maps);
      case 4: return launch_tb<Est, 16, 4>(p, est, g, s, maps);
      case 8: return launch_tb<Est, 16, 8>(p, est, g, s, maps);
      case 16: return launch_tb<Est, 16, 16>(p, est, g, s, maps);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  if (p.env_width == 32) {
    switch (p.width) {
      case 1: return launch_tb<Est, 32, 1>(p, est, g, s, maps);
      case 2: return launch_tb<Est, 32, 2>(p, est, g, s, maps);
      case 4: return launch_tb<Est, 32, 4>(p, est, g, s, maps);
      case 8: return launch_tb<Est, 32, 8>(p, est, g, s, maps);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  return cudaErrorInvalidConfiguration;
}

template <class Est>
static cudaError_t launch_tf_any(const Plan& p, const Est& est, const Geom& g, cudaStream_t s) {
  if (p.env_width == 32) {
    switch (p.width) {
      case 1: return launch_tf<Est, 32, 1>(p, est, g, s);
      case 2: return launch_tf<Est, 32, 2>(p, est, g, s);
      case 4: return launch_tf<Est, 32, 4>(p, est, g, s);
      case 8: return launch_tf<Est, 32, 8>(p, est, g, s);
      case 16: return launch_tf<Est, 32, 16>(p, est, g, s);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  if constexpr (sizeof(typename Est::Store) == 2) {
    // 2-byte storage: 16 environments make a 32-byte sector of a step row
    if (p.env_width == 16) {
      switch (p.width) {
        case 2: return launch_tf<Est, 16, 2>(p, est, g, s);
        case 4: return launch_tf<Est, 16, 4>(p, est, g, s);
        case 8: return launch_tf<Est, 16, 8>(p, est, g, s);
        case 16: return launch_tf<Est, 16, 16>(p, est, g, s);
        case 32: return launch_tf<Est, 16, 32>(p, est, g, s);
        default: return cudaErrorInvalidConfiguration;
      }
    }
  }
  if (p.env_width == 8) {
    switch (p.width) {
      case 4: return launch_tf<Est, 8, 4>(p, est, g, s);
      case 8: return launch_tf<Est, 8, 8>(p, est, g, s);
      case 16: return launch_tf<Est, 8, 16>(p, est, g, s);
      case 32: return launch_tf<Est, 8, 32>(p, est, g, s);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  return cudaErrorInvalidConfiguration;
}

template <class Est>
static cudaError_t launch_pass(const Plan& p, const Est& est, const Geom& g, cudaStream_t s, const TmaSet& maps) {
  if (p.fast) {
    switch (p.width) {
      case 1: return launch_fast_w<Est, 1>(p, est, g, s);
      case 2: return launch_fast_w<Est, 2>(p, est, g, s);
      case 4: return launch_fast_w<Est, 4>(p, est, g, s);
      case 8: return launch_fast_w<Est, 8>(p, est, g, s);
      case 16: return launch_fast_w<Est, 16>(p, est, g, s);
      case 32: return launch_fast_w<Est, 32>(p, est, g, s);
      case 64: return launch_fast_w<Est, 64>(p, est, g, s);
      case 128: return launch_fast_w<Est, 128>(p, est, g, s);
      case 256: return launch_fast_w<Est, 256>(p, est, g, s);
      case 512: return launch_fast_w<Est, 512>(p, est, g, s);
      case 1024: return launch_fast_w<Est, 1024>(p, est, g, s);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  if (p.tm_bulk) return launch_tb_any(p, est, g, s, maps);
  if (p.tm_fast) return p.tm_staged ? launch_ts_any(p, est, g, s) : launch_tf_any(p, est, g, s);
  if (p.time_major) {
    switch (p.width) {
      case 1: return launch_tm_c<Est, 1>(p, est, g, s);
      case 2: return launch_tm_c<Est, 2>(p, est, g, s);
      case 4: return launch_tm_c<Est, 4>(p, est, g, s);
      case 8: return launch_tm_c<Est, 8>(p, est, g, s);
      case 16: return launch_tm_c<Est, 16>(p, est, g, s);
      case 32: return launch_tm_c<Est, 32>(p, est, g, s);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  switch (p.width) {
    case 1: return launch_em_w<Est, 1>(p, est, g, s);
    case 2: return launch_em_w<Est, 2>(p, est, g, s);
    case 4: return launch_em_w<Est, 4>(p, est, g, s);
    case 8: return launch_em_w<Est, 8>(p, est, g, s);
    case 16: return launch_em_w<Est, 16>(p, est, g, s);
    case 32: return launch_em_w<Est, 32>(p, est, g, s);
    case 64: return launch_em_w<Est, 64>(p, est, g, s);
    case 128: return launch_em_w<Est, 128>(p, est, g, s);
    case 256: return launch_em_w<Est, 256>(p, est, g, s);
    case 512: return launch_em_w<Est, 512>(p, est, g, s);
    case 1024: return launch_em_w<Est, 1024>(p, est, g, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

// Retrace's second pass on the fast time-major driver where the plan
// allows it (retrace_tail_plan); false: not taken, the caller runs the
// first pass's kernel again
template <class Est>
static bool launch_retrace_tail(const Est&, const Plan&, const Geom&, cudaStream_t, cudaError_t*) {
  return false;
}
template <bool H, class ST>
static bool launch_retrace_tail(const RetraceEst<H, ST>& est, const Plan& p, const Geom& g, cudaStream_t s,
                                cudaError_t* err) {
  Plan q;
  if (g.aux == nullptr || !retrace_tail_plan(p, g.E, g.T, sizeof(ST) == 2, &q)) return false;
  RetraceTailEst<H, ST> tail;
  tail.b = est.b;
  tail.r = est.r;
  tail.aux = g.aux;
  tail.plane = g.E * (int64_t)g.T;
  tail.out = est.out;
  tail.gamma = est.gamma;
  if constexpr (sizeof(ST) == 2) {
    switch (q.width) {
      case 2: *err = launch_tf<RetraceTailEst<H, ST>, 16, 2>(q, tail, g, s); return true;
      case 4: *err = launch_tf<RetraceTailEst<H, ST>, 16, 4>(q, tail, g, s); return true;
      case 8: *err = launch_tf<RetraceTailEst<H, ST>, 16, 8>(q, tail, g, s); return true;
      case 16: *err = launch_tf<RetraceTailEst<H, ST>, 16, 16>(q, tail, g, s); return true;
      case 32: *err = launch_tf<RetraceTailEst<H, ST>, 16, 32>(q, tail, g, s); return true;
      default: return false;
    }
  } else {
    switch (q.width) {
      case 4: *err = launch_tf<RetraceTailEst<H, ST>, 8, 4>(q, tail, g, s); return true;
      case 8: *err = launch_tf<RetraceTailEst<H, ST>, 8, 8>(q, tail, g, s); return true;
      case 16: *err = launch_tf<RetraceTailEst<H, ST>, 8, 16>(q, tail, g, s); return true;
      case 32: *err = launch_tf<RetraceTailEst<H, ST>, 8, 32>(q, tail, g, s); return true;
      default: return false;
    }
  }
}

template <class Est>
cudaError_t run_scan(const Est& est, const Plan& p, const Geom& g0, cudaStream_t s) {
  TmaSet maps;  // filled for the bulk driver only (the other drivers never read it)
  if constexpr (Est::kStageable) {
    if (p.tm_bulk) {
      maps = TmaSet{};
      StagedList in;
      est.staged_io(in);
      if (!encode_tm_maps(in, (int)sizeof(typename Est::Store), g0.E, g0.T, p.env_width, p.tile, &maps))
        return cudaErrorInvalidValue;
    }
  }
  Geom g = g0;
  if (p.nseg > 1) {
    g.mode = kModeAggregate;
    cudaError_t e = launch_pass(p, est, g, s, maps);
    if (e != cudaSuccess) return e;
    g.mode = kModeFull;
    if (launch_retrace_tail(est, p, g, s, &e)) return e;
  }
  g.mode = kModeFull;
  return launch_pass(p, est, g, s, maps);
}

// The device status word of the kernels of the translation unit that
// includes this header (tma.cuh): ORed into *word, zeroed with clear.
static cudaError_t tu_status(unsigned int* word, bool clear) {
  unsigned int w = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&w, g_tu_status, sizeof(w));
  if (e != cudaSuccess) return e;
  *word |= w;
  if (clear && w != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_tu_status, &zero, sizeof(zero));
  }
  return e;
}

}  // namespace rlca
