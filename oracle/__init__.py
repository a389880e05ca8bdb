"""CPU oracles of the RT-Lynx layer (test infrastructure only; never imported by the library).

``oracle.cpp``         the plain C++ oracle (``lynx_oracle.cpp``, std::thread row split): the reference of the
                       GPU parity tests and the timed CPU baseline;
``oracle.lynx_oracle`` the float64 numpy oracle, kept as an independent cross-check of the C++ one.

Both are pinned by ``tests/test_oracle_pins.py``.
"""
