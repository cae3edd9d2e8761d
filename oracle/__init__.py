"""fp64 CPU oracle for the fused decode-attention block.

TEST INFRASTRUCTURE: imported only by ``tests/``, ``__graft_entry__.smoke()``
and the CPU baseline leg of ``bench.py``. It shares no code with the CUDA
library under ``out_proj_block_gb300/``.
"""
