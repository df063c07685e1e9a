"""GB300-native speculative Whisper decoding (block drafter + block verify).

The compute lives in ``libws.so`` (hand-written CUDA for sm_103a) behind the
C ABI of ``include/ws.h``.  ``binding`` marshals arguments to it through
ctypes and ``runtime`` drives the propose / verify / accept loop.  Importing
``binding`` fails when the library has not been built: there is no CPU path.
"""
__all__ = ["binding", "runtime"]
