"""CPU oracle for the paged-KV hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product package.
The oracle shares no code with the CUDA path; see ``oracle.c`` for the
definitions it transcribes and the passages they follow.
"""
