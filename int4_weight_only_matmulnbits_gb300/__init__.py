"""GB300 (sm_103a) weight-only INT4 blockwise MatMul, MatMulNBits form.

The computation lives in the C-ABI library libmnb.so (include/mnb.h); this
package is its thin Python binding plus the seeded workload generators. The
library is loaded on first use and its absence is an error.
"""
from .binding import (EXPORTS, MNB_CODES_AFFINE, MNB_CODES_CODEBOOK, ChainOp, MnbChain,
                      MnbError, MnbGraph, PackedHeaderC, PackedWeight, library_path, load,
                      mnb_chain_build, mnb_chain_run, mnb_chain_run_noalloc,
                      mnb_fault_status, mnb_graph_build, mnb_matmul, mnb_matmul_bnb4, mnb_matmul_from_host,
                      mnb_matmul_gate_up, mnb_matmul_grouped, mnb_matmul_plan,
                      mnb_matmul_rmsnorm, mnb_matmul_workspace, mnb_packed_forget,
                      mnb_packed_header_make, mnb_packed_read_header, mnb_packed_register,
                      mnb_prepack, mnb_prepack_bnb4, mnb_prepack_qdq, mnb_prepacked_sizes,
                      mnb_set_programmatic_launch, mnb_test_wait_fault, mnb_unprepack,
                      mnb_version, status_string)
from ._build import build_library

__all__ = ["EXPORTS", "MNB_CODES_AFFINE", "MNB_CODES_CODEBOOK", "ChainOp", "MnbChain",
           "MnbError", "MnbGraph", "PackedHeaderC", "PackedWeight", "build_library", "library_path",
           "load", "mnb_chain_build", "mnb_chain_run", "mnb_chain_run_noalloc",
           "mnb_fault_status", "mnb_graph_build", "mnb_matmul", "mnb_matmul_bnb4", "mnb_matmul_from_host",
           "mnb_matmul_gate_up", "mnb_matmul_grouped", "mnb_matmul_plan", "mnb_matmul_rmsnorm",
           "mnb_matmul_workspace", "mnb_packed_forget", "mnb_packed_header_make",
           "mnb_packed_read_header", "mnb_packed_register", "mnb_prepack", "mnb_prepack_bnb4",
           "mnb_prepack_qdq", "mnb_prepacked_sizes", "mnb_set_programmatic_launch",
           "mnb_test_wait_fault",
           "mnb_unprepack", "mnb_version", "status_string"]
