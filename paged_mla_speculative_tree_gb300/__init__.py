"""GB300 (sm_103a) MLA tree-verify attention over a paged bf16 latent KV pool.

The compute path is the CUDA library built from ``csrc/`` behind the C ABI in
``include/mla_tree_verify.h``; ``binding`` is its ctypes binding and
``workloads`` draws seeded synthetic inputs.
"""
from .binding import (MlaTreeVerify, MtvError, MtvPlan, choose_nsplit, clear_device_error, load,  # noqa: F401
                      plan, read_device_error, read_static_device_error, run, run_static, strerror)
