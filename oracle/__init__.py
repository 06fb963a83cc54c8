"""CPU oracle for paged KV gather/scatter -- test infrastructure only (see kv_oracle.py)."""
from .kv_oracle import (LAYER_MAJOR, STRIPE_ALIGN, STRIPED, TOKEN_MAJOR, Chunk, Pool, Request,
                        build, chunk_bytes, load, moved_bytes, store)

__all__ = ["LAYER_MAJOR", "STRIPE_ALIGN", "STRIPED", "TOKEN_MAJOR", "Chunk", "Pool", "Request",
           "build", "chunk_bytes", "load", "moved_bytes", "store"]
