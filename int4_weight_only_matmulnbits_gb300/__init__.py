"""GB300 (sm_103a) weight-only INT4 blockwise MatMul, MatMulNBits form.

The computation lives in the C-ABI library libmnb.so (include/mnb.h); this
package is its thin Python binding plus the seeded workload generators. The
library is loaded on first use and its absence is an error.
"""
from .binding import (EXPORTS, ChainOp, MnbChain, MnbError, PackedWeight, load,
                      library_path, mnb_chain_build, mnb_chain_run,
                      mnb_chain_run_noalloc, mnb_matmul_rmsnorm,
                      mnb_prepack_bnb4, mnb_matmul_bnb4,
                      mnb_fault_status, mnb_matmul, mnb_matmul_from_host,
                      mnb_matmul_workspace, mnb_matmul_plan,
                      mnb_matmul_gate_up, mnb_matmul_grouped, mnb_prepack,
                      mnb_prepack_qdq,
                      mnb_prepacked_sizes, mnb_set_programmatic_launch,
                      mnb_unprepack, mnb_version, status_string)
from ._build import build_library

__all__ = ["EXPORTS", "ChainOp", "MnbChain", "mnb_chain_build", "mnb_chain_run", "mnb_chain_run_noalloc", "mnb_matmul_rmsnorm", "mnb_prepack_bnb4", "mnb_matmul_bnb4", "MnbError", "PackedWeight", "build_library", "load",
           "library_path", "mnb_fault_status", "mnb_matmul", "mnb_matmul_workspace", "mnb_matmul_plan", "mnb_matmul_gate_up", "mnb_matmul_grouped", "mnb_matmul_from_host", "mnb_prepack", "mnb_prepack_qdq",
           "mnb_prepacked_sizes", "mnb_set_programmatic_launch", "mnb_unprepack",
           "mnb_version", "status_string"]
